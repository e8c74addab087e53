// pa_api.cu -- the C ABI (include/pa.h): host-side planning and argument
// checks, the launch of the partition kernel, and the log-sum-exp merge kernel.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <mutex>

#include "pa_common.cuh"

namespace pa {

template <int D, typename E>
cudaError_t launch_attend_d(int G, bool split, const AttendParams& p, dim3 grid,
                            cudaStream_t stream);
template <int D, typename T>
cudaError_t launch_attend_mma_d(bool split, const AttendParams& p, const CUtensorMap* maps,
                                dim3 grid, cudaStream_t stream);
template <int D, typename T>
cudaError_t launch_attend_mma_rope_d(bool split, const AttendParams& p, const CUtensorMap* maps,
                                     dim3 grid, cudaStream_t stream);

template <int D, typename T, bool ROPE>
cudaError_t attend_mma_cluster_occupancy(int c, int* clusters, bool deep);

template <typename T>
static cudaError_t launch_attend_mma_t(int D, bool split, const AttendParams& p,
                                       const CUtensorMap* maps, dim3 grid, cudaStream_t stream) {
    switch (D) {
        case 64: return launch_attend_mma_d<64, T>(split, p, maps, grid, stream);
        case 96: return launch_attend_mma_d<96, T>(split, p, maps, grid, stream);
        case 128: return launch_attend_mma_d<128, T>(split, p, maps, grid, stream);
        case 256: return launch_attend_mma_d<256, T>(split, p, maps, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

static cudaError_t launch_attend_mma(int D, int dtype, bool split, const AttendParams& p,
                                     const CUtensorMap* maps, dim3 grid, cudaStream_t stream) {
    if (p.rope) {
        const bool bf = dtype == PA_DTYPE_BF16;
        switch (D) {
            case 64:
                return bf ? launch_attend_mma_rope_d<64, __nv_bfloat16>(split, p, maps, grid, stream)
                          : launch_attend_mma_rope_d<64, __half>(split, p, maps, grid, stream);
            case 96:
                return bf ? launch_attend_mma_rope_d<96, __nv_bfloat16>(split, p, maps, grid, stream)
                          : launch_attend_mma_rope_d<96, __half>(split, p, maps, grid, stream);
            case 128:
                return bf ? launch_attend_mma_rope_d<128, __nv_bfloat16>(split, p, maps, grid, stream)
                          : launch_attend_mma_rope_d<128, __half>(split, p, maps, grid, stream);
            case 256:
                return bf ? launch_attend_mma_rope_d<256, __nv_bfloat16>(split, p, maps, grid, stream)
                          : launch_attend_mma_rope_d<256, __half>(split, p, maps, grid, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    return dtype == PA_DTYPE_BF16
               ? launch_attend_mma_t<__nv_bfloat16>(D, split, p, maps, grid, stream)
               : launch_attend_mma_t<__half>(D, split, p, maps, grid, stream);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        else
            cudaGetLastError();
    });
    return fn;
}

// The K (or V) cache as a tensor of 16-bit elements for the tensor-core
// kernel's page copies, one copy per page.  D a multiple of 64: 3-D
// [D/64 slabs][rows = num_pages*Hkv*16][64 columns] -- the slab dimension
// outermost (stride 128 bytes) so that the box, 64 x 16 x D/64, lands as the
// page's slabs back to back (16 rows x 128 bytes each) -- with the 128-byte
// swizzle.  D = 96: 3-D [rows][D/32][32], box 32 x D/32 x 16 (a whole page),
// 64-byte swizzle.
static bool make_page_map(CUtensorMap* map, const void* base, long long rows, int D,
                          int dtype) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const CUtensorMapDataType et =
        dtype == PA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (D % 64 == 0) {
        const cuuint64_t dims[3] = {64u, (cuuint64_t)rows, (cuuint64_t)(D / 64)};
        const cuuint64_t strides[2] = {(cuuint64_t)D * 2, 128u};
        const cuuint32_t box[3] = {64u, (cuuint32_t)kPageSize, (cuuint32_t)(D / 64)};
        const cuuint32_t estr[3] = {1, 1, 1};
        return enc(map, et, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
               CUDA_SUCCESS;
    }
    const cuuint64_t dims[3] = {32u, (cuuint64_t)(D / 32), (cuuint64_t)rows};
    const cuuint64_t strides[2] = {64u, (cuuint64_t)D * 2};
    const cuuint32_t box[3] = {32u, (cuuint32_t)(D / 32), (cuuint32_t)kPageSize};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, et, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// make_page_map through a small per-thread cache keyed by every input of the
// encoding (base address, rows, head dim, element type): a map is a pure
// function of them, so a hit is the map the encoder would return.  Decode
// steps reuse the same K/V pools.  Measured on GB300 (Grace host, bursts of
// calls from an idle stream): 1.94 -> 1.75 us of host time per pa_decode, and
// 2.24 -> 1.74 us for a rotary plan together with the cached frequency table
// below.
static bool cached_page_map(CUtensorMap* map, const void* base, long long rows, int D,
                            int dtype) {
    struct Entry {
        alignas(64) CUtensorMap map;
        const void* base;
        long long rows;
        int D, dtype;
        bool valid;
    };
    constexpr int kEntries = 8;
    thread_local Entry cache[kEntries] = {};
    thread_local int next = 0;
    for (int i = 0; i < kEntries; ++i) {
        const Entry& e = cache[i];
        if (e.valid && e.base == base && e.rows == rows && e.D == D && e.dtype == dtype) {
            *map = e.map;
            return true;
        }
    }
    if (!make_page_map(map, base, rows, D, dtype)) return false;
    Entry& e = cache[next];
    next = (next + 1) % kEntries;
    e.map = *map;
    e.base = base;
    e.rows = rows;
    e.D = D;
    e.dtype = dtype;
    e.valid = true;
    return true;
}

// Clusters of c CTAs that one wave holds, with per_sm resident CTAs on each
// of num_sms SMs, for a plan made for an explicit SM count (no device is
// asked).  A cluster must fit inside one GPC, so part of the slots stay
// unused.  The tables are cudaOccupancyMaxActiveClusters of the tensor-core
// kernel measured on GB300 (152 SMs) at 2 and 3 CTAs per SM, for c = 1..16;
// other SM counts use the smaller of the two tables' fill fractions.  A plan
// for the current device (num_sms = 0) asks the device instead
// (device_clusters_per_wave).
static long long clusters_per_wave(int num_sms, int per_sm, int c) {
    static const short k2[kMaxClusterParts] = {304, 152, 97, 74, 58, 46, 38, 36,
                                               30,  28,  23, 23, 19, 14, 14, 14};
    static const short k3[kMaxClusterParts] = {456, 228, 148, 110, 87, 74, 59, 51,
                                               46,  43,  36,  36,  28, 26, 26, 21};
    if (c < 1 || c > kMaxClusterParts) return 0;
    if (num_sms == 152 && per_sm == 2) return k2[c - 1];
    if (num_sms == 152 && per_sm == 3) return k3[c - 1];
    const double f = std::min(k2[c - 1] * (double)c / 304.0, k3[c - 1] * (double)c / 456.0);
    return (long long)((double)num_sms * per_sm * f / c);
}

// cudaOccupancyMaxActiveClusters of the cluster-merge instance for (head
// dim, element type, rotary, deep rings) and clusters of c CTAs on the
// current device, queried once per device and cached; -1 if the query fails.
static long long device_clusters_per_wave(int D, int dtype, bool rope, int c, bool deep = false) {
    constexpr int kMaxDevices = 64;
    static std::atomic<int> cache[kMaxDevices][4][2][2][2][kMaxClusterParts];  // value + 1; 0 = unknown
    int dev = 0;
    if (c < 2 || c > kMaxClusterParts || cudaGetDevice(&dev) != cudaSuccess || dev < 0 ||
        dev >= kMaxDevices) {
        cudaGetLastError();
        return -1;
    }
    const int di = D == 64 ? 0 : D == 96 ? 1 : D == 128 ? 2 : 3;
    const int ti = dtype == PA_DTYPE_BF16 ? 1 : 0;
    std::atomic<int>& slot = cache[dev][di][ti][rope ? 1 : 0][deep ? 1 : 0][c - 1];
    const int known = slot.load();
    if (known > 0) return known - 1;
    int n = 0;
    cudaError_t e = cudaErrorInvalidValue;
#define PA_OCC(DD, TT, RR) e = attend_mma_cluster_occupancy<DD, TT, RR>(c, &n, deep)
#define PA_OCC_D(TT, RR)                                                          \
    switch (D) {                                                                  \
        case 64: PA_OCC(64, TT, RR); break;                                       \
        case 96: PA_OCC(96, TT, RR); break;                                       \
        case 128: PA_OCC(128, TT, RR); break;                                     \
        default: PA_OCC(256, TT, RR); break;                                      \
    }
    if (ti) {
        if (rope) { PA_OCC_D(__nv_bfloat16, true) } else { PA_OCC_D(__nv_bfloat16, false) }
    } else {
        if (rope) { PA_OCC_D(__half, true) } else { PA_OCC_D(__half, false) }
    }
#undef PA_OCC_D
#undef PA_OCC
    if (e != cudaSuccess || n < 0) {
        cudaGetLastError();
        return -1;
    }
    slot.store(n + 1);
    return n;
}

// CTAs of the partition kernel resident per SM (the launch bound, which the
// configurations' static checks also guarantee in shared memory), for G query
// heads per CTA.
int attend_ctas_per_sm(int kernel, int dtype, int D, int G, bool rope) {
    if (kernel == PA_KERNEL_MMA && rope) {
        switch (D) {
            case 64: return MmaCfg<64, true>::kMinBlocks;
            case 96: return MmaCfg<96, true>::kMinBlocks;
            case 128: return MmaCfg<128, true>::kMinBlocks;
            default: return MmaCfg<256, true>::kMinBlocks;
        }
    }
    if (kernel == PA_KERNEL_MMA) {
        switch (D) {
            case 64: return MmaCfg<64>::kMinBlocks;
            case 96: return MmaCfg<96>::kMinBlocks;
            case 128: return MmaCfg<128>::kMinBlocks;
            default: return MmaCfg<256>::kMinBlocks;
        }
    }
    const bool f32 = dtype == PA_DTYPE_F32;
    switch (D) {
        case 64: return f32 ? AttendCfg<64, 4>::blocks_for(G) : AttendCfg<64>::blocks_for(G);
        case 128: return f32 ? AttendCfg<128, 4>::blocks_for(G) : AttendCfg<128>::blocks_for(G);
        default: return f32 ? AttendCfg<256, 4>::blocks_for(G) : AttendCfg<256>::blocks_for(G);
    }
}

// Pages a sequence can attend: ceil(Lmax / ps), or with a window at most
// ceil((window - 1) / ps) + 1 (the window need not start on a page edge).
static int attended_span_pages(int max_context_len, int window) {
    int span = (max_context_len + kPageSize - 1) / kPageSize;
    if (window > 0) {
        const int wspan = (window - 1 + kPageSize - 1) / kPageSize + 1;
        if (wspan < span) span = wspan;
    }
    return span < 1 ? 1 : span;
}

// CTAs per (KV head, head chunk) of a work-balanced plan, or 0 where none can
// be made: the tensor-core kernel without rotary embedding (its rotary
// instances are built without the run-time mapping), B <= kMaxBalancedBatch, one wave of
// resident CTAs over all groups (filled to a little under its slots), the
// last-CTA merge able to stage G x X partials, and partitions of at most
// kMaxStagedPages pages for any lengths within the plan's bound
// (ceil(B * span / (X - B)) <= kMaxStagedPages).
static int balanced_ctas(int kernel, int dtype, int D, int G, bool rope, int batch,
                         int groups_per_seq, int span, int num_sms) {
    if (kernel != PA_KERNEL_MMA || rope || batch < 1 || batch > kMaxBalancedBatch) return 0;
    const long long slots = (long long)num_sms * attend_ctas_per_sm(kernel, dtype, D, G, rope);
    const long long fill = slots - slots / 64;
    long long x = fill / groups_per_seq;
    x = std::min<long long>(x, kFusedMaxStaged / G);
    x = std::min<long long>(x, kMaxPartitions);
    if (x <= batch) return 0;
    if ((long long)batch * span > (long long)kMaxStagedPages * (x - batch)) return 0;
    return (int)x;
}

template <typename E>
static cudaError_t launch_attend_e(int D, int G, bool split, const AttendParams& p, dim3 grid,
                                   cudaStream_t stream) {
    switch (D) {
        case 64: return launch_attend_d<64, E>(G, split, p, grid, stream);
        case 128: return launch_attend_d<128, E>(G, split, p, grid, stream);
        case 256: return launch_attend_d<256, E>(G, split, p, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_attend(int D, int G, bool split, const AttendParams& p, dim3 grid,
                          cudaStream_t stream) {
    switch (p.dtype) {
        case PA_DTYPE_F32: return launch_attend_e<float>(D, G, split, p, grid, stream);
        case PA_DTYPE_BF16: return launch_attend_e<__nv_bfloat16>(D, G, split, p, grid, stream);
        default: return launch_attend_e<__half>(D, G, split, p, grid, stream);
    }
}

// ---------------------------------------------------------------------------
// Log-sum-exp merge of the partition partials (the Phase 2 reduction of the
// paged_attention_v2_pytorch.py commit note):
//   M = max_p m_p,  w_p = 2^(m_p - M) * l_p,  Lambda = sum_p w_p
//   out = sum_p w_p * o_p / Lambda,  lse = (M + log2 Lambda) * ln 2
// with m in the log2 domain and o_p already divided by its own exp-sum l_p.
// Grid (Hq, B, D / 64): a CTA serves 64 output dims of one (head, sequence)
// with 16 float4 columns x 8 partition groups, reduced across groups in
// shared memory; small CTAs with many loads each keep three CTAs per SM, so
// the grid of a long-context step fits in one wave.  Launched with programmatic stream serialization: its CTAs
// may become resident while the partition kernel drains, and wait for it with
// griddepcontrol.wait before touching the workspace.
// ---------------------------------------------------------------------------
constexpr int kMergeThreads = 128;
constexpr int kMergeCols = 16;                          // float4 columns per CTA (64 dims)
constexpr int kMergeGroups = kMergeThreads / kMergeCols;  // partition groups (8)

__device__ __forceinline__ float block_reduce(float v, float* red, bool is_max) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int mask = 16; mask > 0; mask >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, mask);
        v = is_max ? fmaxf(v, o) : v + o;
    }
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    v = red[0];
    for (int w = 1; w < kMergeThreads / 32; ++w) v = is_max ? fmaxf(v, red[w]) : v + red[w];
    return v;
}

template <typename T>
__device__ __forceinline__ T to_elem(float v);
template <>
__device__ __forceinline__ __half to_elem<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 to_elem<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}
template <>
__device__ __forceinline__ float to_elem<float>(float v) { return v; }

template <typename T>
__global__ void __launch_bounds__(kMergeThreads, 3) merge_kernel(const MergeParams p) {
    // Partitions are taken in chunks of kChunk; within a chunk every load (the
    // chunk's m and l, and each thread's kPer float4 slices of o) is issued
    // before any is used, so a chunk costs one memory round trip.  Chunks are
    // combined with a running maximum (the same log-sum-exp algebra).
    constexpr int kPer = 32;
    constexpr int kChunk = kMergeGroups * kPer;  // 256 partitions
    constexpr int kMlPer = kChunk / kMergeThreads;  // (m, l) pairs per thread per chunk
    __shared__ float s_w[kChunk];
    __shared__ float s_red[32];
    __shared__ __align__(16) float s_acc[kMergeGroups][kMergeCols * 4];

    const int h = blockIdx.x;
    const int b = blockIdx.y;
    const int D = p.D;
    const int d0 = blockIdx.z * (kMergeCols * 4);
    const size_t bh = (size_t)b * p.Hq + h;
    const size_t row0 = bh * p.P;
    allow_dependent_launch();  // the next call's partition grid may be scheduled now
    wait_for_prerequisite_grid();
    // A work-balanced plan: the partition size the partition kernel chose from
    // the lengths, which it left in the workspace's info block.
    const int pages_per_part = p.balanced ? *p.ws_info : p.pages_per_part;
    const SeqSpan sp = seq_span(p.context_lens[b], p.window, p.max_ctx, p.maxp, pages_per_part);
    T* orow = reinterpret_cast<T*>(p.out) + bh * D + d0;
    const int ncols = min(kMergeCols * 4, D - d0);  // a 96-dim head ends in a half chunk
    if (!sp.valid) {
        if (threadIdx.x == 0 && h == 0 && blockIdx.z == 0) atomicOr(p.err, PA_DEVERR_BAD_LENGTH);
        if (threadIdx.x < ncols) orow[threadIdx.x] = to_elem<T>(NAN);
        if (threadIdx.x == 0 && blockIdx.z == 0) p.lse[bh] = NAN;
        return;
    }
    const int np = sp.num_parts;
    if (np == 0) {
        if (threadIdx.x < ncols) orow[threadIdx.x] = to_elem<T>(0.f);
        if (threadIdx.x == 0 && blockIdx.z == 0) p.lse[bh] = -INFINITY;
        return;
    }
    const int grp = threadIdx.x / kMergeCols;
    const int col = (threadIdx.x % kMergeCols) * 4;
    const bool col_ok = col < ncols;
    const float* src = p.ws_o + row0 * D + d0 + (col_ok ? col : 0);

    float M = -INFINITY;   // running max (log2 domain)
    float lam = 0.f;       // running sum of partition weights
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < np; c0 += kChunk) {
        float m_i[kMlPer], l_i[kMlPer];
#pragma unroll
        for (int u = 0; u < kMlPer; ++u) {
            const int i_ml = c0 + threadIdx.x + u * kMergeThreads;
            m_i[u] = i_ml < np ? p.ws_m[row0 + i_ml] : -INFINITY;
            l_i[u] = i_ml < np ? p.ws_l[row0 + i_ml] : 0.f;
        }
        float4 o[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = c0 + grp + k * kMergeGroups;
            o[k] = (col_ok && i < np) ? *reinterpret_cast<const float4*>(src + (size_t)i * D)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mloc = m_i[0];
#pragma unroll
        for (int u = 1; u < kMlPer; ++u) mloc = fmaxf(mloc, m_i[u]);
        const float Mc = block_reduce(mloc, s_red, true);
        const float Mn = fmaxf(M, Mc);
        const float rescale = (M == -INFINITY) ? 0.f : ex2(M - Mn);
        float wloc = 0.f;
#pragma unroll
        for (int u = 0; u < kMlPer; ++u) {
            // l == 0 marks a partition with nothing attended; a NaN (a
            // partition that met a bad page) is kept so that it reaches the
            // output.
            const float w = (l_i[u] == 0.f) ? 0.f : ex2(m_i[u] - Mn) * l_i[u];
            s_w[threadIdx.x + u * kMergeThreads] = w;
            wloc += w;
        }
        const float wsum = block_reduce(wloc, s_red, false);  // also orders the s_w writes
        lam = lam * rescale + wsum;
        acc.x *= rescale;
        acc.y *= rescale;
        acc.z *= rescale;
        acc.w *= rescale;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = grp + k * kMergeGroups;
            const float wk = (c0 + i < np) ? s_w[i] : 0.f;
            acc.x += wk * o[k].x;
            acc.y += wk * o[k].y;
            acc.z += wk * o[k].z;
            acc.w += wk * o[k].w;
        }
        M = Mn;
        __syncthreads();  // s_w is rewritten by the next chunk
    }
    *reinterpret_cast<float4*>(&s_acc[grp][col]) = acc;
    __syncthreads();
    const float inv = 1.f / lam;
    if (threadIdx.x < ncols) {
        float a = 0.f;
#pragma unroll
        for (int g = 0; g < kMergeGroups; ++g) a += s_acc[g][threadIdx.x];
        orow[threadIdx.x] = to_elem<T>(a * inv);
    }
    if (threadIdx.x == 0 && blockIdx.z == 0) p.lse[bh] = (M + log2f(lam)) * 0.69314718055994531f;
}

cudaError_t launch_merge(int D, const MergeParams& p, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.Hq, p.B, (D + kMergeCols * 4 - 1) / (kMergeCols * 4));
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    switch (p.dtype) {
        case PA_DTYPE_BF16: return cudaLaunchKernelEx(&cfg, merge_kernel<__nv_bfloat16>, p);
        case PA_DTYPE_F32: return cudaLaunchKernelEx(&cfg, merge_kernel<float>, p);
        default: return cudaLaunchKernelEx(&cfg, merge_kernel<__half>, p);
    }
}

// Workspace layout: [control block | arrival counters (one per group) |
// m (B*Hq*R) | l (B*Hq*R) | o (B*Hq*R*D)], each region 256-byte aligned, for
// R partials per head (partials_per_head; none when P = 1).  The control
// block's first word is the device error word; it and the counters
// (ctrl_bytes in all) must start at zero and are left at zero by every call.
struct WsLayout {
    size_t ctr_off, ctrl_bytes, info_off, m_off, l_off, o_off, total;
};

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// groups = B * Hkv * head chunks (one arrival counter each).  balanced: a
// work-balanced plan, whose partition kernel leaves the partition size it
// chose in a 256-byte info block behind the control bytes for the merge
// kernel (it need not be zero and is not part of ctrl_bytes).
static WsLayout ws_layout(int B, int Hq, int D, int P, int R, long long groups,
                          bool balanced = false) {
    WsLayout w;
    w.ctr_off = kCtrlBytes;
    if (P <= 1) {
        w.ctrl_bytes = w.info_off = w.m_off = w.l_off = w.o_off = kCtrlBytes;
        w.total = kCtrlBytes;
        return w;
    }
    const size_t rows = (size_t)B * Hq * R;
    w.ctrl_bytes = kCtrlBytes + align256((size_t)groups * 4);
    w.info_off = w.ctrl_bytes;
    w.m_off = w.info_off + (balanced ? 256 : 0);
    w.l_off = w.m_off + align256(rows * 4);
    w.o_off = w.l_off + align256(rows * 4);
    w.total = w.o_off + align256(rows * D * 4);
    return w;
}

}  // namespace pa

using namespace pa;

extern "C" {

int pa_version(void) { return (0 << 16) | 1; }

const char* pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported configuration";
        case PA_ERR_CUDA: return "CUDA error";
        case PA_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

int pa_plan(int batch, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
            int num_pages, int max_pages_per_seq, int max_context_len, int window,
            int partition_size, int num_sms, pa_plan_t* plan) {
    return pa_plan_ex(batch, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                      max_pages_per_seq, max_context_len, window, partition_size, num_sms,
                      PA_DTYPE_F16, 0, 0.f, plan);
}

int pa_plan_ex(int batch, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
               int num_pages, int max_pages_per_seq, int max_context_len, int window,
               int partition_size, int num_sms, int dtype, int kernel, float rope_theta,
               pa_plan_t* plan) {
    if (!plan) return PA_ERR_INVALID_ARG;
    memset(plan, 0, sizeof(*plan));
    if (dtype != PA_DTYPE_F16 && dtype != PA_DTYPE_BF16 && dtype != PA_DTYPE_F32)
        return PA_ERR_INVALID_ARG;
    if (!(rope_theta >= 0.f) || rope_theta == INFINITY) return PA_ERR_INVALID_ARG;
    // The tensor-core kernel's rotary instances: fp16 and bf16, every head dim.
    const bool mma_rope_ok = dtype != PA_DTYPE_F32;
    if (kernel == 0)  // automatic: fp32, and rotary embeddings the tensor-core kernel lacks, need the CUDA-core kernel
        kernel = (dtype == PA_DTYPE_F32 || (rope_theta > 0.f && !mma_rope_ok)) ? PA_KERNEL_SIMT
                                                                               : PA_KERNEL_MMA;
    if (kernel != PA_KERNEL_SIMT && kernel != PA_KERNEL_MMA) return PA_ERR_INVALID_ARG;
    if (kernel == PA_KERNEL_MMA && (dtype == PA_DTYPE_F32 || (rope_theta > 0.f && !mma_rope_ok)))
        return PA_ERR_UNSUPPORTED;
    if (kernel == PA_KERNEL_SIMT && head_dim == 96)
        return PA_ERR_UNSUPPORTED;
    if (batch < 0 || batch > 65535 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_q_heads % num_kv_heads != 0 || head_dim <= 0 || page_size <= 0 || num_pages <= 0 ||
        max_pages_per_seq <= 0 || max_context_len < 0 || window < 0 ||
        (partition_size < 0 && partition_size != PA_PARTITION_BALANCED) || num_sms < 0)
        return PA_ERR_INVALID_ARG;
    if ((long long)max_context_len > (long long)max_pages_per_seq * page_size)
        return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 96 && head_dim != 128 && head_dim != 256)
        return PA_ERR_UNSUPPORTED;
    if (page_size != kPageSize) return PA_ERR_UNSUPPORTED;
    bool want_balanced = partition_size == PA_PARTITION_BALANCED;
    if (want_balanced) partition_size = 0;
    bool auto_split = false;  // the automatic plan is a whole-wave fixed split
    if (partition_size % page_size != 0) return PA_ERR_INVALID_ARG;

    const int g = num_q_heads / num_kv_heads;
    const int nchunk = (g + kMaxHeadsPerCta - 1) / kMaxHeadsPerCta;
    if (g % nchunk != 0) return PA_ERR_UNSUPPORTED;
    const int G = g / nchunk;
    if ((long long)num_kv_heads * nchunk > 65535) return PA_ERR_UNSUPPORTED;

    const bool this_device = num_sms == 0;  // plan for the current device: ask it
    if (num_sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return PA_ERR_CUDA;
        }
    }

    const int span = attended_span_pages(max_context_len, window);
    // Work-balanced partitions: X CTAs per (KV head, head chunk), one wave
    // over all groups, when the batch's pages always fit X partitions.
    const int bal_x = balanced_ctas(kernel, dtype, head_dim, G, rope_theta > 0.f, batch,
                                    num_kv_heads * nchunk, span, num_sms);
    if (want_balanced && bal_x == 0) return PA_ERR_UNSUPPORTED;

    int pp;  // pages per partition
    bool use_cluster = false;
    if (partition_size > 0) {
        pp = partition_size / page_size;
    } else {
        // Automatic: split only when it pays.  A group's whole context of at
        // most kNoSplitBytes streams through one CTA faster than a second
        // launch (the merge) costs, and when the unsplit grid already fills
        // the GPU a split only adds merge traffic.  Otherwise cut each group's
        // span so that the grid is a whole number of waves of resident CTAs
        // (the fewest waves whose partitions fit kMaxPagesPerPart), with at
        // least kMinPagesPerPart pages per partition.
        constexpr long long kNoSplitBytes = 128 << 10;
        constexpr int kMinPagesPerPart = 2 * kWarps;
        const long long groups = (long long)batch * num_kv_heads * nchunk;
        const long long slots = (long long)num_sms * attend_ctas_per_sm(kernel, dtype, head_dim, G, rope_theta > 0.f);
        // A wave is filled to a little under its slots: a grid that needs
        // every slot measured slow at 3 CTAs per SM (head dims 64 and 128,
        // B = 1: 456 CTAs 92.5 us, 448 CTAs 81.6 us per step on GB300) and
        // no faster at 2 per SM.  The partition kernel alone runs the same
        // either way; the merge kernel's CTAs, resident early under
        // programmatic dependent launch, leave a full grid short of slots.
        const long long fill = slots - slots / 64;
        const long long span_bytes =
            (long long)span * 2 * page_size * head_dim * (dtype == PA_DTYPE_F32 ? 4 : 2);
        // Cluster merge (tensor-core kernel): the largest cluster C (2 ..
        // kMaxClusterParts) of which one wave holds one per group, when the
        // span cut C ways gives short partitions (at most
        // kClusterMaxPagesPerPart pages).  The grid is then that single wave
        // and the merge stays on chip.  Longer partitions keep the
        // whole-wave split below: a cluster wave leaves slots empty and some
        // SMs with more CTAs than others, which costs more there than the
        // merge launch saves (measured on GB300).
        constexpr int kClusterMaxPagesPerPart = 64;
        long long cpar = 0;
        const int per_sm = attend_ctas_per_sm(kernel, dtype, head_dim, G, rope_theta > 0.f);
        for (int c = kMaxClusterParts; c >= 2 && groups > 0; --c) {
            long long held = -1;
            if (this_device && kernel == PA_KERNEL_MMA)
                held = device_clusters_per_wave(head_dim, dtype, rope_theta > 0.f, c);
            if (held < 0) held = clusters_per_wave(num_sms, per_sm, c);
            if (held >= groups) {
                cpar = c;
                break;
            }
        }
        const int cpp = cpar >= 2 ? std::max<int>((int)((span + cpar - 1) / cpar), kMinPagesPerPart) : 0;
        if (groups == 0 || groups >= slots || span_bytes <= kNoSplitBytes) {
            pp = span;
        } else if (kernel == PA_KERNEL_MMA && cpar >= 2 && cpp <= kClusterMaxPagesPerPart &&
                   (span + cpp - 1) / cpp >= 2) {
            pp = cpp;
            use_cluster = true;
        } else {
            pp = span;
            for (long long waves = 1; waves <= 64; ++waves) {
                long long parts = waves * fill / groups;
                if (parts < 1) parts = 1;
                pp = (int)((span + parts - 1) / parts);
                if (pp <= kMaxPagesPerPart) break;
            }
            if (pp < kMinPagesPerPart) pp = kMinPagesPerPart;
            auto_split = true;
        }
        if (pp > kMaxPagesPerPart) pp = kMaxPagesPerPart;
    }
    // A batch of several sequences whose automatic plan is a fixed split
    // takes work-balanced partitions instead: the host knows only the bound
    // on the lengths, and a split sized for it leaves the CTAs of short
    // sequences idle while the long ones stream.  Measured on GB300 (32 query
    // / 8 KV heads, head dim 128): lengths {100, 200, 300, 50000} 54.7 ->
    // 39.1 us, {100000, 500, 800, 20} 82.1 -> 68.4 us, eight lengths up to
    // 64K 174.4 -> 170.9 us; uniform lengths lose 1-2 % (4 x 100000: 236.0 ->
    // 240.5 us).  Short contexts keep the cluster merge: the last-CTA merge
    // that balanced plans use costs about 2 us more than it.
    if (!want_balanced && partition_size == 0 && auto_split && batch >= 2 && bal_x > 0)
        want_balanced = true;
    if (want_balanced) {
        // the largest partition any lengths within max_context_len can give
        pp = (int)(((long long)batch * span + (bal_x - batch) - 1) / (bal_x - batch));
        pp = std::max(kMinBalancedPages, std::min(pp, kMaxStagedPages));
        use_cluster = false;
    }
    if (pp > (kernel == PA_KERNEL_MMA ? kMaxStagedPages : kMaxPagesPerPart))
        return PA_ERR_UNSUPPORTED;
    const int P = want_balanced ? bal_x : (span + pp - 1) / pp;
    if (P > kMaxPartitions) return PA_ERR_UNSUPPORTED;

    plan->batch = batch;
    plan->num_q_heads = num_q_heads;
    plan->num_kv_heads = num_kv_heads;
    plan->head_dim = head_dim;
    plan->page_size = page_size;
    plan->num_pages = num_pages;
    plan->max_pages_per_seq = max_pages_per_seq;
    plan->max_context_len = max_context_len;
    plan->window = window;
    plan->partition_size = pp * page_size;
    plan->num_partitions = P;
    plan->heads_per_cta = G;
    plan->num_sms = num_sms;
    const long long groups_all = (long long)batch * num_kv_heads * nchunk;
    // Sized for one partial per partition, the most any parts_per_cta needs,
    // so that a caller may lower parts_per_cta in this plan.
    const WsLayout wl = ws_layout(batch, num_q_heads, head_dim, P, P, groups_all, want_balanced);
    plan->workspace_bytes = wl.total;
    plan->ctrl_bytes = (int)wl.ctrl_bytes;
    plan->kernel = kernel;
    plan->dtype = dtype;
    plan->rope_theta = rope_theta;
    // Merge inside the partition kernel when a group's partials are small
    // (its last CTA merges them, no second launch); the merge kernel when they
    // are many (the one-CTA merge would then trail the grid).
    plan->cluster = (use_cluster && P >= 2 && P <= kMaxClusterParts) ? P : 0;
    // Deep page rings for cluster grids that do not fill the GPU (head dims
    // 96, 128 and 256 without rotary embedding; the others have one
    // instance): with at most one CTA per SM each CTA streams alone, and more
    // pages in flight per warp win.  Measured on GB300 (graph-timed, default
    // vs deep instance): 32/8 heads at D 128, one sequence of 16K tokens
    // 18.0 vs 16.1 us, of 8K 11.15 vs 10.43 us, two of 8K 14.4 vs 14.0 us; a
    // full grid (8 ragged sequences) 14.3 vs 15.6 us.  At D 256 the deep
    // instance runs 1 CTA per SM with 6-page rings: one sequence of 16K
    // tokens, 24/4 heads (64 CTAs) 18.9 vs 17.05 us, but 128 CTAs (8/4 heads,
    // two sequences; or 16/8 heads) 10.6 vs 16.2 and 15.6 vs 21.6 us, so
    // there it is taken only for grids of at most half the SMs.
    plan->deep_ring = 0;
    if (plan->cluster > 1 && kernel == PA_KERNEL_MMA && rope_theta <= 0.f &&
        (head_dim == 96 || head_dim == 128 || head_dim == 256)) {
        const long long groups = (long long)batch * num_kv_heads * nchunk;
        const int deep_per_sm = head_dim == 256 ? 1 : 2;
        const long long max_ctas = head_dim == 256 ? num_sms / 2 : num_sms;
        if (groups * plan->cluster <= max_ctas) {
            long long held = -1;
            if (this_device) held = device_clusters_per_wave(head_dim, dtype, false, plan->cluster, true);
            if (held < 0) held = clusters_per_wave(num_sms, deep_per_sm, plan->cluster);
            if (held >= groups) plan->deep_ring = 1;
        }
    }
    // Tensor-core kernel: each warp's first two pages are requested into L2
    // before the dependency wait.  Measured on GB300: 0.4-1.5 us less per
    // step when decode steps follow each other with programmatic dependent
    // launch; 0.5-1 us more per call behind a kernel that does not launch
    // dependents early (a caller in that case sets 0).
    plan->prewait_prefetch = kernel == PA_KERNEL_MMA ? 2 : 0;
    plan->merge_in_kernel =
        (kernel == PA_KERNEL_MMA && P > 1 && plan->cluster == 0 && kFusedMergeFits(G, head_dim, P))
            ? 1
            : 0;
    // Rotary instances (fixed partitions): the last CTA of each group merges
    // whenever a group's partials are at most 128 KiB.  Measured on GB300
    // (graph-timed, last CTA vs merge kernel): 4 x 32K tokens, 32/8 heads,
    // D 128, P 9: 96.1 vs 97.4 us; 24/4 heads, D 256, P 18 (110 KB): 99.9 vs
    // 103.6 us.  The same 24/4-head shape without rotary embedding is faster
    // with the merge kernel (82.6 vs 84.9 us), so the rule is for these
    // instances only.
    if (kernel == PA_KERNEL_MMA && rope_theta > 0.f && P > 1 && plan->cluster == 0 &&
        (long long)P * G * head_dim * 4 <= (128 << 10) && kFusedMergeLegal(G, head_dim, P))
        plan->merge_in_kernel = 1;
    plan->balanced = want_balanced ? bal_x : 0;
    if (want_balanced) {
        // The merge of a balanced plan: the last CTA of each group, unless a
        // group can leave it too much to merge alone -- one sequence taking
        // all but B - 1 of the X CTAs, X - B + 1 partials of G x D floats --
        // when the merge kernel, which spreads a group over many CTAs, wins.
        // Measured on GB300 (graph-timed, last CTA vs merge kernel): 24/4
        // heads at D 256 with one long sequence 51.5 vs 44.5 us (442 KB
        // worst case), 64/8 heads at D 128 43.1 vs 40.8 us (217 KB); 16
        // sequences, 32/8 heads at D 128 16.4 vs 22.4 us (84 KB), 32/8 heads
        // at D 96 66.9 vs 67.2 us (81 KB).
        constexpr long long kLastCtaMergeMaxBytes = 128 << 10;
        const long long worst = (long long)(bal_x - batch + 1) * G * head_dim * 4;
        plan->merge_in_kernel = worst <= kLastCtaMergeMaxBytes ? 1 : 0;
    }
    // Partitions per CTA (tensor-core kernel, split plans without a
    // cluster): a CTA may serve 2 or 4 consecutive partitions and merge them
    // into one partial, which cuts CTA prologues and epilogues, the partials
    // written and the merge's reads.  Measured on GB300 (1, 2 and 4 per CTA
    // over batches 1-16, head dims 64-256, 32K-128K tokens): a grid of just
    // over one wave of resident CTAs is the slow case (its last wave runs a
    // few CTAs alone, 1.1-1.3 waves measured 3-12 % slower), while one wave
    // that still covers every SM, or 1.5 waves and more, run fast.  So keep
    // one partition per CTA when that grid already fits in one wave (filled
    // to a little under its slots, as above), and otherwise take the largest
    // of 4 and 2 whose grid is either.
    {
        const long long groups = (long long)batch * num_kv_heads * nchunk;
        const long long slots = (long long)num_sms *
                                attend_ctas_per_sm(kernel, dtype, head_dim, G, rope_theta > 0.f);
        const long long fill = slots - slots / 64;
        int ppc = 1;  // (the CUDA-core kernel always serves one)
        if (kernel == PA_KERNEL_MMA && plan->cluster == 0 && !plan->balanced && slots > 0 &&
            P >= 2 && groups * P > fill) {
            for (int c = 4; c >= 2; c /= 2) {
                if (c > P || (long long)c * pp > kMaxPagesPerPart) continue;
                const long long n = groups * ((P + c - 1) / c);
                if ((n >= num_sms && n <= fill) || 2 * n >= 3 * slots) {
                    ppc = c;
                    break;
                }
            }
        }
        plan->parts_per_cta = ppc;
    }
    const long long ctas =
        plan->balanced ? (long long)plan->balanced * num_kv_heads * nchunk
                       : (long long)((P + plan->parts_per_cta - 1) / plan->parts_per_cta) *
                             num_kv_heads * nchunk * batch;
    plan->ctas = (int)std::min<long long>(ctas, INT_MAX);
    return PA_OK;
}

// Partitions per partial row: the tensor-core kernel merges the
// parts_per_cta partitions of a CTA into one partial; the CUDA-core kernel
// writes one per partition.
static int parts_per_partial(const pa_plan_t* plan) {
    return (plan->kernel == PA_KERNEL_MMA && plan->num_partitions > 1) ? plan->parts_per_cta : 1;
}

// Partial rows per (sequence, query head): one per CTA along the partitions.
static int partials_per_head(const pa_plan_t* plan) {
    const int c = parts_per_partial(plan);
    return (plan->num_partitions + c - 1) / c;
}

static int check_plan(const pa_plan_t* plan) {
    if (!plan) return PA_ERR_INVALID_ARG;
    const int B = plan->batch, Hq = plan->num_q_heads, Hkv = plan->num_kv_heads;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || plan->page_size != kPageSize ||
        plan->num_partitions < 1 || plan->num_partitions > kMaxPartitions ||
        plan->partition_size < kPageSize || plan->partition_size % kPageSize != 0 ||
        plan->num_pages <= 0 ||
        plan->max_pages_per_seq <= 0 || plan->max_context_len < 0 || plan->window < 0)
        return PA_ERR_INVALID_ARG;
    if (plan->head_dim != 64 && plan->head_dim != 96 && plan->head_dim != 128 &&
        plan->head_dim != 256)
        return PA_ERR_UNSUPPORTED;
    if (plan->dtype != PA_DTYPE_F16 && plan->dtype != PA_DTYPE_BF16 &&
        plan->dtype != PA_DTYPE_F32)
        return PA_ERR_INVALID_ARG;
    if (!(plan->rope_theta >= 0.f) || plan->rope_theta == INFINITY) return PA_ERR_INVALID_ARG;
    // Rotary embedding: the CUDA-core kernel (fp16, fp32), or the tensor-core
    // kernel's rotary instances (fp16, bf16), which keep
    // the rotated q and K as head + remainder pairs.
    // The CUDA-core kernel is built for fp16/bf16/fp32 and head dims
    // 64/128/256; the tensor-core kernel for fp16/bf16 and head dims 64/96/128/256.
    if (plan->kernel == PA_KERNEL_SIMT && plan->head_dim == 96)
        return PA_ERR_UNSUPPORTED;
    if (plan->kernel == PA_KERNEL_MMA && plan->dtype == PA_DTYPE_F32) return PA_ERR_UNSUPPORTED;
    const int g = Hq / Hkv;
    const int G = plan->heads_per_cta;
    if (G < 1 || G > kMaxHeadsPerCta || g % G != 0) return PA_ERR_INVALID_ARG;
    if (plan->kernel != PA_KERNEL_SIMT && plan->kernel != PA_KERNEL_MMA) return PA_ERR_INVALID_ARG;
    if (plan->parts_per_cta < 1) return PA_ERR_INVALID_ARG;
    const int R = partials_per_head(plan);
    const WsLayout wl = ws_layout(B, Hq, plan->head_dim, plan->num_partitions, R,
                                  (long long)B * Hkv * (Hq / Hkv / plan->heads_per_cta),
                                  plan->balanced > 0);
    if (plan->workspace_bytes < wl.total) return PA_ERR_INVALID_ARG;
    // The control bytes a caller keeps zero must cover the error word and
    // every arrival counter this plan's launch uses (a plan edited after
    // pa_plan, e.g. a different heads_per_cta, may need more of them).
    if (plan->ctrl_bytes < 0 || (size_t)plan->ctrl_bytes < wl.ctrl_bytes ||
        (size_t)plan->ctrl_bytes > plan->workspace_bytes)
        return PA_ERR_INVALID_ARG;
    if (plan->merge_in_kernel && !kFusedMergeLegal(plan->heads_per_cta, plan->head_dim, R))
        return PA_ERR_INVALID_ARG;
    if (plan->balanced < 0) return PA_ERR_INVALID_ARG;
    if (plan->balanced > 0) {
        // Work-balanced partitions: one partition per CTA, no cluster, one
        // load of all B lengths per CTA, and no partition longer than
        // kMaxStagedPages for lengths within the plan's bound.  Either merge:
        // the last CTA of each group, or the merge kernel (which works out
        // the same partition size from the lengths).
        const int X = plan->balanced;
        const int span = attended_span_pages(plan->max_context_len, plan->window);
        if (plan->kernel != PA_KERNEL_MMA || plan->cluster > 1 ||
            plan->parts_per_cta != 1 || B > kMaxBalancedBatch || X <= B ||
            plan->num_partitions != X || plan->rope_theta > 0.f ||
            (long long)B * span > (long long)kMaxStagedPages * (X - B))
            return PA_ERR_INVALID_ARG;
    }
    if (plan->cluster < 0) return PA_ERR_INVALID_ARG;
    if (plan->deep_ring != 0 && plan->deep_ring != 1) return PA_ERR_INVALID_ARG;
    if (plan->deep_ring == 1 && plan->cluster > 1 &&
        (plan->kernel != PA_KERNEL_MMA || plan->rope_theta > 0.f ||
         (plan->head_dim != 96 && plan->head_dim != 128 && plan->head_dim != 256)))
        return PA_ERR_INVALID_ARG;
    if (plan->prewait_prefetch < 0 || plan->prewait_prefetch > kMaxPrewaitPrefetch)
        return PA_ERR_INVALID_ARG;
    if (plan->test_stall_bytes < 0 || plan->test_stall_bytes > 4096) return PA_ERR_INVALID_ARG;
    if (plan->cluster > 1 &&
        (plan->kernel != PA_KERNEL_MMA || plan->cluster > kMaxClusterParts ||
         plan->num_partitions != plan->cluster || plan->parts_per_cta != 1 ||
         plan->merge_in_kernel))
        return PA_ERR_INVALID_ARG;
    // Page ids a CTA stages: kMaxStagedPages (tensor-core kernel) or
    // kMaxPagesPerPart (CUDA-core kernel) for its parts_per_cta partitions.
    const int staged = plan->kernel == PA_KERNEL_MMA ? kMaxStagedPages : kMaxPagesPerPart;
    if (plan->parts_per_cta < 1 ||
        (long long)plan->parts_per_cta * (plan->partition_size / kPageSize) > staged)
        return PA_ERR_INVALID_ARG;
    // The tensor-core kernel gives each of a CTA's partitions 4 / parts_per_cta warps.
    if (plan->kernel == PA_KERNEL_MMA && plan->parts_per_cta != 1 && plan->parts_per_cta != 2 &&
        plan->parts_per_cta != 4)
        return PA_ERR_INVALID_ARG;
    // TMA row coordinates are signed 32-bit.
    if (plan->kernel == PA_KERNEL_MMA &&
        (long long)plan->num_pages * Hkv * kPageSize > 0x7fffffffLL)
        return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int pa_decode_partitions(const pa_plan_t* plan, const void* q, const void* k_cache,
                         const void* v_cache, const int32_t* block_tables,
                         const int32_t* context_lens, float scale, int window, void* out,
                         float* lse, void* workspace, void* stream) {
    int st = check_plan(plan);
    if (st != PA_OK) return st;
    if (window != plan->window) return PA_ERR_INVALID_ARG;
    if (!workspace) return PA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PA_ERR_INVALID_ARG;
    if (plan->batch == 0) return PA_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !lse)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return PA_ERR_INVALID_ARG;

    const int D = plan->head_dim;
    const int P = plan->num_partitions;
    const int R = partials_per_head(plan);
    const int nchunk = plan->num_q_heads / plan->num_kv_heads / plan->heads_per_cta;
    const WsLayout wl = ws_layout(plan->batch, plan->num_q_heads, D, P, R,
                                  (long long)plan->batch * plan->num_kv_heads * nchunk,
                                  plan->balanced > 0);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    AttendParams p;
    p.q = static_cast<const __half*>(q);
    p.k = static_cast<const __half*>(k_cache);
    p.v = static_cast<const __half*>(v_cache);
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = static_cast<__half*>(out);
    p.lse = lse;
    p.ws_m = reinterpret_cast<float*>(ws + wl.m_off);
    p.ws_l = reinterpret_cast<float*>(ws + wl.l_off);
    p.ws_o = reinterpret_cast<float*>(ws + wl.o_off);
    p.err = reinterpret_cast<unsigned*>(ws);
    p.counters = reinterpret_cast<unsigned*>(ws + wl.ctr_off);
    p.ws_info = reinterpret_cast<int*>(ws + wl.info_off);
    p.merge_in_kernel = (plan->kernel == PA_KERNEL_MMA && P > 1 && plan->merge_in_kernel) ? 1 : 0;
    p.cluster = (plan->kernel == PA_KERNEL_MMA && P > 1 && plan->cluster > 1) ? plan->cluster : 0;
    p.deep = p.cluster > 1 && plan->deep_ring == 1 ? 1 : 0;
    p.B = plan->batch;
    p.Hq = plan->num_q_heads;
    p.Hkv = plan->num_kv_heads;
    p.g = plan->num_q_heads / plan->num_kv_heads;
    p.num_pages = plan->num_pages;
    p.maxp = plan->max_pages_per_seq;
    p.max_ctx = plan->max_context_len;
    p.window = plan->window;
    p.P = R;  // partial rows per head: one per CTA along x
    p.pages_per_part = plan->partition_size / kPageSize;
    p.nchunk = p.g / plan->heads_per_cta;
    p.heads_per_cta = plan->heads_per_cta;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    p.rope = plan->rope_theta > 0.f ? 1 : 0;
    p.dtype = plan->dtype;
    if (p.rope) {
        // theta_i / (2 pi) in double, split into two floats; the table of the
        // last (base, head dim) this thread used is kept.
        thread_local float t_base = 0.f;
        thread_local int t_D = 0;
        thread_local float t_phi[2][kMaxRopePairs];
        if (t_base != plan->rope_theta || t_D != D) {
            for (int i = 0; i < D / 2; ++i) {
                const double turn = pow((double)plan->rope_theta, -2.0 * i / D) / (2.0 * M_PI);
                const float hi = (float)turn;
                t_phi[0][i] = hi;
                t_phi[1][i] = (float)(turn - (double)hi);
            }
            t_base = plan->rope_theta;
            t_D = D;
        }
        memcpy(p.rope_phi[0], t_phi[0], sizeof(float) * (D / 2));
        memcpy(p.rope_phi[1], t_phi[1], sizeof(float) * (D / 2));
    }
    cudaError_t e;
    if (plan->kernel == PA_KERNEL_MMA) {
        alignas(64) CUtensorMap maps[2];  // K, V
        const long long rows = (long long)plan->num_pages * p.Hkv * kPageSize;
        if (!cached_page_map(&maps[0], k_cache, rows, D, plan->dtype) ||
            !cached_page_map(&maps[1], v_cache, rows, D, plan->dtype))
            return PA_ERR_CUDA;
        p.parts_per_cta = P > 1 ? plan->parts_per_cta : 1;  // one partition: all warps on it
        p.prewait_prefetch = plan->prewait_prefetch;
        p.stall_tx = plan->test_stall_bytes;
        p.balanced = plan->balanced;
        // A work-balanced plan spreads the batch over grid.x (X CTAs per group).
        const dim3 grid = plan->balanced
                              ? dim3(plan->balanced, p.Hkv * p.nchunk, 1)
                              : dim3((P + p.parts_per_cta - 1) / p.parts_per_cta,
                                     p.Hkv * p.nchunk, p.B);
        e = launch_attend_mma(D, plan->dtype, P > 1, p, maps, grid,
                              static_cast<cudaStream_t>(stream));
    } else {
        p.parts_per_cta = 1;
        p.prewait_prefetch = 0;
        p.stall_tx = 0;
        p.balanced = 0;
        const dim3 grid(P, p.Hkv * p.nchunk, p.B);
        e = launch_attend(D, plan->heads_per_cta, P > 1, p, grid,
                          static_cast<cudaStream_t>(stream));
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

int pa_merge(const pa_plan_t* plan, const int32_t* context_lens, void* out, float* lse,
             void* workspace, void* stream) {
    int st = check_plan(plan);
    if (st != PA_OK) return st;
    if (!workspace) return PA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PA_ERR_INVALID_ARG;
    if (plan->batch == 0 || plan->num_partitions == 1) return PA_OK;
    // The partition kernel already merged (in its last CTAs, or in each cluster).
    if (plan->kernel == PA_KERNEL_MMA && (plan->merge_in_kernel || plan->cluster > 1)) return PA_OK;
    if (!context_lens || !out || !lse || !aligned16(out)) return PA_ERR_INVALID_ARG;
    const int D = plan->head_dim;
    const int nchunk = plan->num_q_heads / plan->num_kv_heads / plan->heads_per_cta;
    const int R = partials_per_head(plan);
    const WsLayout wl = ws_layout(plan->batch, plan->num_q_heads, D, plan->num_partitions, R,
                                  (long long)plan->batch * plan->num_kv_heads * nchunk,
                                  plan->balanced > 0);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    MergeParams p;
    p.context_lens = context_lens;
    p.ws_m = reinterpret_cast<const float*>(ws + wl.m_off);
    p.ws_l = reinterpret_cast<const float*>(ws + wl.l_off);
    p.ws_o = reinterpret_cast<const float*>(ws + wl.o_off);
    p.out = out;
    p.lse = lse;
    p.err = reinterpret_cast<unsigned*>(ws);
    p.ws_info = reinterpret_cast<const int*>(ws + wl.info_off);
    p.B = plan->batch;
    p.Hq = plan->num_q_heads;
    p.D = D;
    // Partial i covers parts_per_cta consecutive partitions from partition
    // i * parts_per_cta on.
    p.P = R;
    p.pages_per_part = (plan->partition_size / kPageSize) * parts_per_partial(plan);
    p.maxp = plan->max_pages_per_seq;
    p.max_ctx = plan->max_context_len;
    p.window = plan->window;
    p.dtype = plan->dtype;
    p.balanced = plan->balanced;
    if (launch_merge(D, p, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

int pa_decode(const pa_plan_t* plan, const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, const int32_t* context_lens, float scale, int window,
              void* out, float* lse, void* workspace, void* stream) {
    int st = pa_decode_partitions(plan, q, k_cache, v_cache, block_tables, context_lens, scale,
                                  window, out, lse, workspace, stream);
    if (st != PA_OK) return st;
    return pa_merge(plan, context_lens, out, lse, workspace, stream);
}

int pa_get_error(void* workspace, void* stream, int* device_error) {
    if (!workspace || !device_error) return PA_ERR_INVALID_ARG;
    unsigned v = 0;
    const int st = pa_get_error_ex(workspace, stream, 0, &v);
    if (st == PA_OK) *device_error = (int)v;
    return st;
}

int pa_get_error_ex(void* workspace, void* stream, int clear, unsigned* device_error) {
    if (!workspace || !device_error) return PA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    *device_error = v;
    if (clear) {
        if (cudaMemsetAsync(workspace, 0, sizeof(unsigned), s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess) {
            cudaGetLastError();
            return PA_ERR_CUDA;
        }
    }
    return PA_OK;
}

}  // extern "C"

namespace pa {
// check_plan, then the extent of the workspace the plan's launches touch:
// its control bytes (error word and arrival counters, which must be zero
// before a call) and its total bytes.  Host only; nothing is launched.
int plan_workspace_extent(const pa_plan_t* plan, size_t* ctrl_bytes, size_t* total_bytes) {
    const int st = check_plan(plan);
    if (st != PA_OK) return st;
    const int nchunk = plan->num_q_heads / plan->num_kv_heads / plan->heads_per_cta;
    const WsLayout wl = ws_layout(plan->batch, plan->num_q_heads, plan->head_dim,
                                  plan->num_partitions, partials_per_head(plan),
                                  (long long)plan->batch * plan->num_kv_heads * nchunk,
                                  plan->balanced > 0);
    *ctrl_bytes = wl.ctrl_bytes;
    *total_bytes = wl.total;
    return PA_OK;
}
}  // namespace pa
