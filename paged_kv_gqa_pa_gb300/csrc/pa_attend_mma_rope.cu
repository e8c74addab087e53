// Tensor-core partition-kernel instances with the rotary embedding (fp16
// caches, head dims 64, 96 and 128), in a translation unit of their own so the
// build compiles them in parallel with the plain instances.
#include "pa_attend_mma.cuh"

namespace pa {
template cudaError_t launch_attend_mma_rope_d<64>(bool, const AttendParams&, const CUtensorMap*,
                                                  dim3, cudaStream_t);
template cudaError_t launch_attend_mma_rope_d<96>(bool, const AttendParams&, const CUtensorMap*,
                                                  dim3, cudaStream_t);
template cudaError_t launch_attend_mma_rope_d<128>(bool, const AttendParams&, const CUtensorMap*,
                                                   dim3, cudaStream_t);
}  // namespace pa
