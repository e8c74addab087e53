// Tensor-core partition-kernel instances, bf16 caches, every head dim (the
// head-group size is a runtime value: the group always fills the n = 8 mma
// columns).  One translation unit per element type so the build compiles them
// in parallel.
#include "pa_attend_mma.cuh"

namespace pa {
template cudaError_t launch_attend_mma_d<64, __nv_bfloat16>(bool, const AttendParams&, const CUtensorMap*,
                                                  dim3, cudaStream_t);
template cudaError_t launch_attend_mma_d<96, __nv_bfloat16>(bool, const AttendParams&, const CUtensorMap*,
                                                  dim3, cudaStream_t);
template cudaError_t launch_attend_mma_d<128, __nv_bfloat16>(bool, const AttendParams&, const CUtensorMap*,
                                                   dim3, cudaStream_t);
template cudaError_t launch_attend_mma_d<256, __nv_bfloat16>(bool, const AttendParams&, const CUtensorMap*,
                                                   dim3, cudaStream_t);
template cudaError_t attend_mma_cluster_occupancy<64, __nv_bfloat16, false>(int, int*, bool);
template cudaError_t attend_mma_cluster_occupancy<96, __nv_bfloat16, false>(int, int*, bool);
template cudaError_t attend_mma_cluster_occupancy<128, __nv_bfloat16, false>(int, int*, bool);
template cudaError_t attend_mma_cluster_occupancy<256, __nv_bfloat16, false>(int, int*, bool);
}  // namespace pa
