// pa_static.cu -- pa_decode_static: pa_decode without a caller workspace.
//
// Some callers cannot allocate device memory at the moment they decode:
// engines and plugins that are handed only the input and output buffers they
// own and have no allocator of their own to draw on, and latency-critical
// loops that must never enter the allocator (cudaMalloc can synchronise the
// device and stall every stream).  For them the partition partials live in a
// fixed scratch array compiled into the library instead of a workspace the
// caller provides.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds PA_STATIC_WORKSPACE_BYTES of it until the process exits.  Its
// name is only a host-side stand-in: the device address is looked up with
// cudaGetSymbolAddress, once per device, on the first call made on that
// device (with that device current), and cached.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/pa.h"

namespace {

__device__ __align__(256) unsigned char g_static_workspace[PA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_static_ptr[kMaxDevices];

// Device address of g_static_workspace on the current device, or nullptr.
void* static_workspace_ptr() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_static_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess || !ptr) {
            cudaGetLastError();
            return nullptr;
        }
        g_static_ptr[dev] = ptr;
    }
    return g_static_ptr[dev];
}

}  // namespace

extern "C" int pa_decode_static(const pa_plan_t* plan, const void* q, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables,
                                const int32_t* context_lens, float scale, int window, void* out,
                                float* lse, void* stream) {
    if (!plan) return PA_ERR_INVALID_ARG;
    if (plan->workspace_bytes > (size_t)PA_STATIC_WORKSPACE_BYTES) return PA_ERR_WORKSPACE;
    void* ws = static_workspace_ptr();
    if (!ws) return PA_ERR_CUDA;
    // The scratch keeps whatever the previous call left in it.  Its control
    // bytes (error word, per-group arrival counters) must start at zero, so
    // they are cleared on the stream before every call: a call that gave up
    // on a bounded wait may have left a counter behind.  The partials need no
    // clearing: each is written before it is read.  cudaMemsetAsync allocates
    // nothing.
    if (plan->batch > 0 && plan->ctrl_bytes > 0 &&
        cudaMemsetAsync(ws, 0, (size_t)plan->ctrl_bytes, static_cast<cudaStream_t>(stream)) !=
            cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return pa_decode(plan, q, k_cache, v_cache, block_tables, context_lens, scale, window, out,
                     lse, ws, stream);
}
