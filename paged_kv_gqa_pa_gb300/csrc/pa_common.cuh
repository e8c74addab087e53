// pa_common.cuh -- shared pieces of the GB300 (sm_103a) paged-KV decode
// kernels: launch parameters, the per-head-dim kernel configuration, and the
// inline-PTX wrappers for mbarriers and 1-D bulk copies (cp.async.bulk).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

constexpr int kPageSize = 16;     // tokens per page
constexpr int kWarps = 4;         // consumer warps per CTA of the attention kernel
constexpr int kThreads = kWarps * 32;
constexpr int kMaxPagesPerPart = 256;  // page ids a CUDA-core CTA stages; the longest
                                       // partition the planner's fixed split makes
constexpr int kMaxStagedPages = 2048;  // page ids a tensor-core CTA stages (in the
                                       // merge scratch, idle while pages stream)
constexpr int kMaxClusterParts = 16;   // largest cluster (the non-portable limit)
constexpr int kMaxPartitions = 4096;   // partitions the merge kernel reduces
constexpr int kMaxHeadsPerCta = 8;
constexpr int kCtrlBytes = 256;        // workspace control block (device error word)
constexpr int kMaxRopePairs = 128;     // head_dim / 2 of the widest rotary head
constexpr int kMaxPrewaitPrefetch = 8; // largest prewait_prefetch (pages per warp)
constexpr int kMinBalancedPages = 2 * kWarps;  // smallest partition of a work-balanced plan
constexpr int kMaxBalancedBatch = kThreads;    // sequences a work-balanced plan can spread
// Partials one (sequence, head chunk) can merge in the last CTA: its G x R
// (m, weight) pairs are staged in the 8 KiB combine buffer.
constexpr int kFusedMaxStaged = 1024;

// Bounded waits: a bulk copy that has not landed after this long is reported
// as PA_DEVERR_TIMEOUT instead of hanging the GPU.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

struct AttendParams {
    const __half* q;
    const __half* k;
    const __half* v;
    const int* block_tables;
    const int* context_lens;
    __half* out;
    float* lse;
    float* ws_o;   // [B, Hq, P, D] partition outputs, normalised by their exp-sum
    float* ws_m;   // [B, Hq, P] partition max, log2 domain
    float* ws_l;   // [B, Hq, P] partition exp-sum
    unsigned* err; // device error word
    unsigned* counters;  // per-(sequence, KV head, head chunk) arrival counters (fused merge)
    int* ws_info;        // work-balanced plans: the partition size chosen, for the merge kernel
    int merge_in_kernel; // 1: the last CTA of each group merges its partials
    int cluster;         // > 1: the group's partitions form one cluster and merge in it
    int deep;            // 1: with a cluster, the deep-ring instance (MmaCfg DEEP; host side)
    int B, Hq, Hkv, g, num_pages, maxp, max_ctx, window;
    int P;                  // partitions (grid.x)
    int pages_per_part;     // partition size in pages
    int nchunk;             // head chunks per KV head (grid.y = Hkv * nchunk)
    int heads_per_cta;      // G: query heads one CTA serves
    int parts_per_cta;      // consecutive partitions one CTA streams (tensor-core kernel)
    int prewait_prefetch;   // pages per warp prefetched into L2 before the PDL wait (tensor-core)
    int balanced;           // > 0: work-balanced partitions over the batch, this many CTAs
                            // along grid.x per (KV head, head chunk) (tensor-core kernel)
    int stall_tx;           // test hook: extra bytes each warp's first copy expects (0 normally)
    float scale_log2;       // scale * log2(e)
    int rope;               // 1: rotary embedding of q and K (CUDA-core kernel)
    int dtype;              // PA_DTYPE_*: q, K, V and out (the CUDA-core kernel's instance)
    // Rotary frequency i as a fraction of a turn, theta_i / (2 pi), split into
    // two floats (rope_phi[0][i] + rope_phi[1][i]) so that pos * theta_i
    // reduces modulo one turn with fp32 accuracy for any position below 2^24.
    float rope_phi[2][kMaxRopePairs];
};

struct MergeParams {
    const int* context_lens;
    const float* ws_o;
    const float* ws_m;
    const float* ws_l;
    const int* ws_info;      // work-balanced plans: the partition size the partition kernel chose
    void* out;               // fp16 or bf16 (dtype)
    float* lse;
    unsigned* err;
    int B, Hq, D, P, pages_per_part, maxp, max_ctx, window;
    int dtype;               // PA_DTYPE_*
    int balanced;            // > 0: work-balanced plan (partition size from the lengths)
};

// Pipeline depth (pages of K or V in flight per warp) for each head dim; the
// resulting shared-memory footprint sets the CTAs per SM.
// (CUDA-core kernel; ES = element bytes: 2 for fp16, 4 for fp32.)
template <int D, int ES = 2>
struct AttendCfg {
    static constexpr int kPageBytes = kPageSize * D * ES;
    static constexpr int kStages =
        ES == 2 ? (D == 256 ? 3 : (D == 128 ? 4 : 6)) : (D == 64 ? 4 : 2);
    static constexpr int kRingBytes = kWarps * kStages * kPageBytes;
    static constexpr int kPBufFloats = kPageSize * kMaxHeadsPerCta * 2;  // per warp: (p, p) pairs
    static constexpr int kSmemBytes = kRingBytes + kWarps * kPBufFloats * 4 +
                                      kMaxPagesPerPart * 4 + kWarps * kMaxHeadsPerCta * 2 * 4 +
                                      kWarps * kStages * 8 + 16;
    static constexpr int kMinBlocks = ES == 2 ? (D == 256 ? 2 : 3) : (D == 256 ? 1 : 3);
    static_assert(kMinBlocks * (kSmemBytes + 1024) <= 228 * 1024, "CTAs per SM by shared memory");
    // The launch bound of the G-head instance: seven or eight heads per CTA
    // keep their q, scores and accumulators in registers only at two CTAs.
    static constexpr int blocks_for(int G) { return (G >= 7 && kMinBlocks > 2) ? 2 : kMinBlocks; }
};

// Tensor-core kernel configuration per head dim (see pa_attend_mma.cuh).
// ROPE: the rotary instances, which keep the rotated q (hi + lo) and the
// lane's rotary state in registers; they run 2 CTAs per SM (3 at D = 64) with
// deeper rings, plus the per-CTA tables of the 8- and 64-token rotations.
// DEEP: the cluster-merge instances of plain head dims 96, 128 and 256 for
// grids that do not fill the GPU: 2 CTAs per SM with the deeper rings (1 with
// 6-page rings at D = 256), since a CTA that streams alone on its SM is bound
// by the bytes its own ring keeps in flight.
template <int D, bool ROPE = false, bool DEEP = false>
struct MmaCfg {
    static_assert(!DEEP || (!ROPE && (D == 96 || D == 128 || D == 256)),
                  "deep rings: plain head dims 96, 128 and 256");
    static_assert(D % 64 == 0 || (D % 64 == 32 && (D / 32) % 2 == 1),
                  "head dim: 64-column slabs, or an odd number of 32-column units");
    static constexpr bool kRows64 = (D % 64) != 0;  // one 3-D box, 64-byte units, 64-byte swizzle
    static constexpr int kFullSlabs = D / 64;       // else: 128-byte slabs (128-byte swizzle)
    static constexpr int kSlabBytes = kPageSize * 128;
    static constexpr int kPageBytes = kPageSize * D * 2;
    // pages in flight per warp; with the fixed buffers below this keeps
    // kMinBlocks CTAs per SM within 228 KiB of shared memory
    static constexpr int kStages = ROPE || DEEP
                                       ? (D == 256 ? (DEEP ? 6 : 3) : (D == 128 ? 6 : (D == 96 ? 8 : 6)))
                                       : (D == 256 ? 3 : (D == 128 ? 4 : (D == 96 ? 5 : 6)));
    static constexpr int kRingBytes = kWarps * kStages * kPageBytes;
    // scratch of the last-CTA merge ((m, weight) pairs of a group's partials);
    // while pages stream it holds the CTA's page ids
    static constexpr int kXBytes = kWarps * kMaxHeadsPerCta * 64 * 4;
    // A CTA combines its warp states at the end, all D dims at once, in the
    // idle page ring behind the cluster partial ([G][D] o, then m and l):
    // rows of D + 4 floats (the pad spreads the four head rows a store writes
    // over distinct banks).
    static constexpr int kWideXOff = ((kMaxHeadsPerCta * D + 2 * kMaxHeadsPerCta) * 4 + 1023) /
                                     1024 * 1024;
    static constexpr int kWideXStride = D + 4;
    static_assert(kWideXOff + kWarps * kMaxHeadsPerCta * kWideXStride * 4 <= kRingBytes,
                  "one-round combine fits in the page ring");
    // rotary tables: (cos, sin) of the 8- and 64-token turns, D/2 frequencies each
    static constexpr int kRopeBytes = ROPE ? 2 * (D / 2) * 8 : 0;
    static_assert(kXBytes >= kMaxStagedPages * 4, "page ids staged in the merge scratch");
    static constexpr int kSmemBytes = 1024 /* alignment slack */ + kRingBytes + kXBytes +
                                      kWarps * kMaxHeadsPerCta * 3 * 4 + kWarps * kStages * 8 +
                                      kRopeBytes + 16;
    static constexpr int kMinBlocks =
        ROPE ? (D == 64 ? 3 : 2) : (DEEP && D == 256 ? 1 : (D == 256 || DEEP ? 2 : 3));
    static_assert(kMinBlocks * (kSmemBytes + 1024) <= 228 * 1024, "CTAs per SM by shared memory");
    static_assert(kRows64 || kPageBytes == kFullSlabs * kSlabBytes, "slab layout");
    static_assert(kPageBytes % 1024 == 0, "page slots keep the 1 KiB swizzle alignment");
};

// The in-kernel merge of the tensor-core kernel issues all of its loads at
// once: kFusedLoads float4 partial slices per thread, plus the (m, l) pairs
// staged in the 8 KiB combine buffer.  It is used only where that covers a
// whole group (G heads x D dims x P partitions) and P is small: measured on
// GB300 it beats the merge kernel for P = 7 and loses to it for P = 19..24,
// where every CTA's fence and arrival lengthen the grid more than the second
// launch costs.
constexpr int kFusedLoads = 24;
constexpr int kFusedMaxParts = 8;

__host__ __device__ constexpr bool kFusedMergeFits(int G, int D, int P) {
    return P <= kFusedMaxParts && G * (D / 4) <= kThreads &&
           (P + (kThreads / (G * (D / 4))) - 1) / (kThreads / (G * (D / 4))) <= kFusedLoads &&
           2 * G * P * 4 <= kWarps * kMaxHeadsPerCta * 64 * 4;
}

// What the last-CTA merge can take at all: the G x R (m, weight) pairs in the
// combine buffer.  Its threads take the (head, 4-dim column) items kThreads at
// a time, and partials beyond kFusedLoads per thread cost one more round trip
// per chunk.
__host__ __device__ constexpr bool kFusedMergeLegal(int G, int D, int R) {
    return D > 0 && G * R <= kFusedMaxStaged;
}
static_assert(2 * kFusedMaxStaged * 4 <= kWarps * kMaxHeadsPerCta * 64 * 4,
              "the staged (m, weight) pairs fit the combine buffer");

// Span of pages a sequence attends, shared by the partition and merge kernels
// so both agree on the partition count of every sequence.
struct SeqSpan {
    int L, start, first_page, end_page, num_parts;
    bool valid;
};

__device__ __forceinline__ SeqSpan seq_span(int L, int window, int max_ctx, int maxp,
                                            int pages_per_part) {
    SeqSpan s;
    s.L = L;
    s.valid = L >= 0 && L <= max_ctx && (L + kPageSize - 1) / kPageSize <= maxp;
    s.start = (window > 0 && window < L) ? L - window : 0;
    s.first_page = s.start / kPageSize;
    s.end_page = (L + kPageSize - 1) / kPageSize;
    const int np = s.valid ? s.end_page - s.first_page : 0;
    s.num_parts = np > 0 ? (np + pages_per_part - 1) / pages_per_part : 0;
    return s;
}

// Sum of v over a CTA of kWarps warps (every thread calls it and gets the
// sum; s_red: kWarps ints of shared memory).
__device__ __forceinline__ int cta_sum(int v, int* s_red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    __syncthreads();  // earlier reads of s_red are done
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    int t = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t += s_red[w];
    return t;
}

// Work-balanced partitions (plan.balanced = X CTAs per (KV head, head chunk)
// over the whole batch).  Thread t < B passes the attended pages of sequence
// t (balanced_seq_pages), every thread gets the partition size pp: the
// smallest with sum_b max(1, ceil(pages_b / pp)) <= X, by bisection between
// ceil(T / X) and ceil(T / (X - B)) (T = sum_b pages_b; the upper end always
// fits since sum_b ceil(pages_b / pp) <= T / pp + B), clamped to
// [kMinBalancedPages, kMaxStagedPages] (the plan guarantees the clamp never
// binds for lengths within its bound).  The partition kernel and the merge
// kernel compute the same pp from the same lengths.
__device__ __forceinline__ int balanced_seq_pages(int L, int window, int max_ctx, int maxp) {
    const SeqSpan sp = seq_span(L, window, max_ctx, maxp, 1);
    return sp.valid ? sp.end_page - sp.first_page : 0;  // (0 for a length out of bounds)
}

__device__ __forceinline__ int balanced_pp(int pages, int B, int X, int* s_red) {
    const int t = threadIdx.x;
    const int T = cta_sum(t < B ? pages : 0, s_red);
    int lo = max(kMinBalancedPages, (T + X - 1) / X);
    int hi = max(lo, min((T + (X - B) - 1) / (X - B), kMaxStagedPages));
    while (lo < hi) {  // (the same bounds in every thread)
        const int mid = (lo + hi) >> 1;
        const int need = cta_sum(t < B ? max(1, (pages + mid - 1) / mid) : 0, s_red);
        if (need <= X)
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo;
}

// ---------------------------------------------------------------------------
// Inline PTX: mbarrier + bulk copy + fast exp2.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Global -> shared bulk copy that signals `bar` with its byte count on arrival.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of `bar`, giving up after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// cos and sin of pos * theta_i for a rotary frequency given as a fraction of a
// turn split into phi1 + phi2: the product is reduced modulo one turn exactly
// (fma recovers the rounding error of pos * phi1), then sincospif evaluates
// the reduced angle.  Accurate to a few fp32 ulps for pos < 2^24.
__device__ __forceinline__ void rope_twiddle(int pos, float phi1, float phi2, float& c,
                                             float& s) {
    const float pf = (float)pos;
    const float hi = pf * phi1;
    const float err = fmaf(pf, phi1, -hi);
    float fr = hi - floorf(hi);
    fr += err + pf * phi2;
    fr -= floorf(fr);
    sincospif(2.f * fr, &s, &c);
}

// 2^x with the MUFU approximation (relative error ~2^-22); -inf -> +0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Request `bytes` (a multiple of 16, 16-byte aligned) of global memory into L2.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Let a dependent grid launched with programmatic stream serialization (the
// merge) get scheduled while this grid's last CTAs still run; the dependent
// grid waits for this grid's completion before it reads anything.
__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the grid this one depends on has completed and its writes are
// visible (no-op for a normal launch).
__device__ __forceinline__ void wait_for_prerequisite_grid() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace pa

// Launchers (pa_attend_d*.cu, pa_attend_mma.cu).
namespace pa {
cudaError_t launch_attend(int D, int G, bool split, const AttendParams& p, dim3 grid,
                          cudaStream_t stream);
int attend_ctas_per_sm(int kernel, int dtype, int D, int G, bool rope);
}  // namespace pa
