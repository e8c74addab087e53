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

namespace pa {
// pa_api.cu: the plan checks of pa_decode, then the control and total bytes
// of the workspace the plan's launches use.
int plan_workspace_extent(const pa_plan_t* plan, size_t* ctrl_bytes, size_t* total_bytes);
}  // namespace pa

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
    // Every check runs on the host before anything touches the GPU: the plan
    // itself (the same rules as pa_decode), then the workspace extent its
    // launches use, worked out from the plan's shapes rather than taken from
    // its ctrl_bytes field, against the size of the built-in array.
    size_t ctrl = 0, total = 0;
    const int st = pa::plan_workspace_extent(plan, &ctrl, &total);
    if (st != PA_OK) return st;
    const size_t cap = (size_t)PA_STATIC_WORKSPACE_BYTES;
    if (plan->workspace_bytes > cap || total > cap || ctrl > cap ||
        (size_t)plan->ctrl_bytes > cap)
        return PA_ERR_WORKSPACE;
    void* ws = static_workspace_ptr();
    if (!ws) return PA_ERR_CUDA;
    // The array keeps whatever the previous call left in it, and that call may
    // have used another plan: its partials may sit where this plan keeps its
    // arrival counters, and its device error word stays set until cleared.
    // So this plan's control bytes are cleared on the stream before every
    // call (cudaMemsetAsync allocates nothing).  The partials need no
    // clearing: each is written before it is read.
    if (plan->batch > 0 &&
        cudaMemsetAsync(ws, 0, ctrl, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return pa_decode(plan, q, k_cache, v_cache, block_tables, context_lens, scale, window, out,
                     lse, ws, stream);
}
