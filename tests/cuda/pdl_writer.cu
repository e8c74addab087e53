// Test helper (not part of the library): a one-CTA kernel that lets the next
// kernel on its stream start early (programmatic dependent launch), waits a
// fixed time, and only then overwrites the block table and the context
// lengths.  A decode launched right after it reads the old values as hints
// before its dependency wait and must use the new ones.  The wait is bounded
// by the global timer: it always ends.
#include <cuda_runtime.h>

__global__ void delayed_copy(const int* src_bt, int* dst_bt, int n_bt, const int* src_cl,
                             int* dst_cl, int n_cl, unsigned long long delay_ns) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    unsigned long long t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    do {
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    } while (t - t0 < delay_ns);
    for (int i = threadIdx.x; i < n_bt; i += blockDim.x) dst_bt[i] = src_bt[i];
    for (int i = threadIdx.x; i < n_cl; i += blockDim.x) dst_cl[i] = src_cl[i];
}

extern "C" int launch_delayed_copy(const int* src_bt, int* dst_bt, int n_bt, const int* src_cl,
                                   int* dst_cl, int n_cl, unsigned long long delay_ns,
                                   void* stream) {
    delayed_copy<<<1, 256, 0, static_cast<cudaStream_t>(stream)>>>(src_bt, dst_bt, n_bt, src_cl,
                                                                    dst_cl, n_cl, delay_ns);
    return (int)cudaGetLastError();
}
