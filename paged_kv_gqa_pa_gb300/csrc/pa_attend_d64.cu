// Partition-kernel instances for head_dim 64 (one translation unit per head dim
// so the build compiles them in parallel).
#include "pa_attend.cuh"

namespace pa {
template cudaError_t launch_attend_d<64>(int, bool, const AttendParams&, dim3, cudaStream_t);
}  // namespace pa
