// Partition-kernel instances for head_dim 256 (one translation unit per head dim
// so the build compiles them in parallel).
#include "pa_attend.cuh"

namespace pa {
template cudaError_t launch_attend_d<256>(int, bool, const AttendParams&, dim3, cudaStream_t);
}  // namespace pa
