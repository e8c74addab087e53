// Tensor-core partition-kernel instances with the rotary embedding (fp16 and
// bf16 caches, head dims 64, 96, 128 and 256), in a translation unit of their own
// so the build compiles them in parallel with the plain instances.
#include "pa_attend_mma.cuh"

namespace pa {
#define PA_ROPE_INSTANCE(D, T)                                                                   \
    template cudaError_t launch_attend_mma_rope_d<D, T>(bool, const AttendParams&,              \
                                                        const CUtensorMap*, dim3, cudaStream_t);
PA_ROPE_INSTANCE(64, __half)
PA_ROPE_INSTANCE(96, __half)
PA_ROPE_INSTANCE(128, __half)
PA_ROPE_INSTANCE(256, __half)
PA_ROPE_INSTANCE(64, __nv_bfloat16)
PA_ROPE_INSTANCE(96, __nv_bfloat16)
PA_ROPE_INSTANCE(128, __nv_bfloat16)
PA_ROPE_INSTANCE(256, __nv_bfloat16)
#undef PA_ROPE_INSTANCE
#define PA_ROPE_OCCUPANCY(D, T) template cudaError_t attend_mma_cluster_occupancy<D, T, true>(int, int*, bool);
PA_ROPE_OCCUPANCY(64, __half)
PA_ROPE_OCCUPANCY(96, __half)
PA_ROPE_OCCUPANCY(128, __half)
PA_ROPE_OCCUPANCY(256, __half)
PA_ROPE_OCCUPANCY(64, __nv_bfloat16)
PA_ROPE_OCCUPANCY(96, __nv_bfloat16)
PA_ROPE_OCCUPANCY(128, __nv_bfloat16)
PA_ROPE_OCCUPANCY(256, __nv_bfloat16)
#undef PA_ROPE_OCCUPANCY
}  // namespace pa
