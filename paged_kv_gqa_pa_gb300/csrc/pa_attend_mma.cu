// Tensor-core partition-kernel instances (all head dims; the head-group size
// is a runtime value because the group always fills the n = 8 mma columns).
#include "pa_attend_mma.cuh"

namespace pa {
template cudaError_t launch_attend_mma_d<64>(bool, const AttendParams&, const CUtensorMap&,
                                             const CUtensorMap&, dim3, cudaStream_t);
template cudaError_t launch_attend_mma_d<128>(bool, const AttendParams&, const CUtensorMap&,
                                              const CUtensorMap&, dim3, cudaStream_t);
template cudaError_t launch_attend_mma_d<256>(bool, const AttendParams&, const CUtensorMap&,
                                              const CUtensorMap&, dim3, cudaStream_t);
}  // namespace pa
