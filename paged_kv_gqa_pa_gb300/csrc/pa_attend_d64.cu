// CUDA-core partition-kernel instances for head_dim 64, fp16 (one translation
// unit per head dim and element type so the build compiles them in parallel).
#include "pa_attend.cuh"

namespace pa {
template cudaError_t launch_attend_d<64, __half>(int, bool, const AttendParams&, dim3,
                                                 cudaStream_t);
}  // namespace pa
