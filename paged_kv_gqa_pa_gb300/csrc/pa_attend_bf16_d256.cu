// CUDA-core partition-kernel instances for head_dim 256, bf16 caches.
#include "pa_attend.cuh"

namespace pa {
template cudaError_t launch_attend_d<256, __nv_bfloat16>(int, bool, const AttendParams&, dim3,
                                                        cudaStream_t);
}  // namespace pa
