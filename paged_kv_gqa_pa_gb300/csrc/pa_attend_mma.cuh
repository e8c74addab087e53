// pa_attend_mma.cuh -- tensor-core variant of the partition kernel.
//
// Same result as attend_kernel (pa_attend.cuh), and the same shape of work: a
// CTA per (partitions, KV head, head chunk, sequence), four warps with their
// own page pipelines, online softmax per page, warp states merged at the end.
// What differs is how a page is staged and contracted, and that a CTA may
// serve several partitions:
//
//  * Staging.  A K or V page arrives through one TMA tensor copy
//    (cp.async.bulk.tensor.3d) of the cache viewed as [D/64 slabs][rows =
//    num_pages*Hkv*16][64 columns] (slab stride 128 bytes, row stride 2D
//    bytes), a box of 64 columns x 16 rows x D/64 slabs, with the 128-byte
//    swizzle: in shared memory the page is its slabs back to back, and the
//    16-byte chunk c of row r of a slab lands at chunk c ^ (r & 7), so the
//    ldmatrix reads below are free of bank conflicts.
//    A head dim that is not a multiple of 64 (96) is copied instead as one
//    3-D box per page, [16 rows][D/32 units of 64 bytes], with the 64-byte
//    swizzle: chunk c of 64-byte unit u (u = row * D/32 + slab) lands at
//    c ^ ((u >> 1) & 3).  D/32 = 3 is odd, so the 8 rows an ldmatrix reads
//    still fall in 8 distinct bank groups.
//  * Element type T: fp16, or bf16 (then q and out are bf16 as well).
//  * q.K (the commit note's Phase 1 QK^T).  S^T[16 tokens x 8 heads] =
//    K_page[16 x D] . Q^T[D x 8] with mma.sync m16n8k16 (fp16 in, fp32
//    accumulate; bf16 in for bf16 caches): K fragments via ldmatrix from the swizzled page, the q
//    fragments sit in registers for the whole CTA.  The group's G <= 8 query
//    heads fill the n = 8 columns (unused columns are zero and never stored).
//  * softmax.  Each lane owns 2 tokens x 2 heads of S^T; page maxima come from
//    three xor-shuffles, exp2 in fp32, and P is rounded to fp16 for the mma.
//    Two exp-sums are kept: of the rounded weights, which normalises the
//    output (so the weights applied to V sum to one), and of the fp32
//    weights, which gives the LSE and the partition's weight in the merge.
//    With bf16 (8 significant bits) P is split into a bf16 head and a bf16
//    remainder, and P.V takes both (two mma per tile), so the weights keep
//    about 16 significant bits.
//  * P.V.  O^T[D x 8] += V^T[D x 16 tokens] . P^T[16 x 8]: V^T fragments via
//    ldmatrix.trans of the same swizzled page, P^T from S^T by movmatrix.trans.
//    The accumulator of a lane holds two heads, so the online rescale needs
//    no data exchange.
//  * Several partitions per CTA.  A CTA may serve parts_per_cta (1, 2 or 4)
//    consecutive partitions of its (sequence, KV head): each partition gets
//    4 / parts_per_cta of the warps, so no warp crosses a partition edge,
//    and at the end, with the page ring idle, one round combines all the
//    CTA's warp states (the merge's log-sum-exp algebra) into one partial
//    row for its partitions together.  Fewer, longer CTAs spend less time in
//    prologues and epilogues, and write and merge fewer partials.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include <atomic>
#include <type_traits>

#include "pa_common.cuh"

namespace pa {

// Element-type specifics: the mma flavour and the packing of fp32 pairs.
template <typename T>
struct Elem;

template <>
struct Elem<__half> {
    __device__ static __forceinline__ void mma(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
            " {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    // (lo, hi) rounded to nearest; the rounded values come back in lo_r, hi_r.
    __device__ static __forceinline__ uint32_t pack2(float lo, float hi, float& lo_r, float& hi_r) {
        __half2 h = __floats2half2_rn(lo, hi);
        const float2 back = __half22float2(h);
        lo_r = back.x;
        hi_r = back.y;
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ static __forceinline__ __half from_float(float v) { return __float2half_rn(v); }
};

template <>
struct Elem<__nv_bfloat16> {
    __device__ static __forceinline__ void mma(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
            " {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    __device__ static __forceinline__ uint32_t pack2(float lo, float hi, float& lo_r, float& hi_r) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        const float2 back = __bfloat1622float2(h);
        lo_r = back.x;
        hi_r = back.y;
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __device__ static __forceinline__ __nv_bfloat16 from_float(float v) {
        return __float2bfloat16_rn(v);
    }
};

template <typename T>
__device__ __forceinline__ void store4(T* dst, float a, float b, float c, float d) {
    float ra, rb, rc, rd;
    uint2 packed;
    packed.x = Elem<T>::pack2(a, b, ra, rb);
    packed.y = Elem<T>::pack2(c, d, rc, rd);
    *reinterpret_cast<uint2*>(dst) = packed;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& a0, uint32_t& a1, uint32_t& a2,
                                        uint32_t& a3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& a0, uint32_t& a1,
                                          uint32_t& a2, uint32_t& a3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Byte offset inside a swizzled page of the 16-byte chunk `chunk` (0..D/8-1)
// of token row `row`.
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    if constexpr (D % 64 == 0) {  // [slab][16 rows][128 bytes], 128-byte swizzle
        return (uint32_t)((chunk >> 3) * (kPageSize * 128) + row * 128 +
                          (((chunk & 7) ^ (row & 7)) << 4));
    } else {  // [16 rows][D/32 units][64 bytes], 64-byte swizzle
        const int unit = row * (D / 32) + (chunk >> 2);
        return (uint32_t)(unit * 64 + (((chunk & 3) ^ ((unit >> 1) & 3)) << 4));
    }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// In-kernel log-sum-exp merge (the commit note's Phase 2) for plans whose
// partials are small: every CTA of a (sequence, KV head, head chunk) group
// that wrote partials arrives on the group's counter once it is done; the
// last one to arrive resets the counter to zero for the next call and merges
// the group's partials (read through L2) into the final fp16 rows and the LSE.
// Nobody waits: a CTA that is not last simply exits.
//
// The merge issues all of its loads at once, so it costs one memory round
// trip: the (m, l) pairs of the G x R partials (R = the group's CTAs that
// attend anything, one partial each), and for each (head, 4-dim
// column) item the partials' o values, spread over kThreads / items threads
// of kFusedLoads loads each.  The planner enables it only where that covers
// the group (kFusedMergeFits).  xbuf holds the G x R (m, weight) pairs, the
// idle page ring the per-thread partial sums.
template <int D, typename T>
__device__ __forceinline__ void group_arrive_and_merge(const AttendParams& p, const SeqSpan& sp,
                                                       int b, int h0, int G, float* xbuf,
                                                       float* s_small, float* scratch) {
    __shared__ int s_last;
    // Arrival: the CTA barrier orders every thread's partial stores before
    // thread 0's arrival, and the arrival is one acquire-release atomic at GPU
    // scope (cumulative, so it releases the whole CTA's stores, and for the
    // last CTA acquires every other CTA's); the closing barrier passes that on
    // to the threads that read the partials.
    __syncthreads();
    if (threadIdx.x == 0) {
        const int target = (sp.num_parts + p.parts_per_cta - 1) / p.parts_per_cta;
        unsigned* ctr = p.counters + ((size_t)b * gridDim.y + blockIdx.y);
        unsigned prev;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                     : "=r"(prev)
                     : "l"(ctr)
                     : "memory");
        const int last = (int)(prev + 1u) == target;
        if (last) atomicExch(ctr, 0u);  // ready for the next call
        s_last = last;
    }
    __syncthreads();
    if (!s_last) return;

    constexpr int D4 = D / 4;
    const int np = (sp.num_parts + p.parts_per_cta - 1) / p.parts_per_cta;  // partials
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int items = G * D4;  // (head, float4 column) pairs
    const size_t row0 = ((size_t)b * p.Hq + h0) * p.P;
    float* s_m = xbuf;           // [G][np]
    float* s_w = xbuf + G * np;  // [G][np]: exp-sums, then merge weights
    float* s_M = s_small;        // [G]
    float* s_L = s_small + kMaxHeadsPerCta;

    // The (m, l) pairs and the first chunk of o slices go out together, so a
    // group of up to kFusedLoads x tpi partials costs one round trip; each
    // further chunk of that many costs one more.  Items are taken kThreads at a
    // time: with fewer items than threads, tpi threads share an item (a
    // stride-tpi slice of the partials each) and add up in shared memory.
    for (int idx = threadIdx.x; idx < G * np; idx += kThreads) {
        const int h = idx / np, i = idx % np;
        s_m[idx] = __ldcg(p.ws_m + row0 + (size_t)h * p.P + i);
        s_w[idx] = __ldcg(p.ws_l + row0 + (size_t)h * p.P + i);
    }
    for (int base = 0; base < items; base += kThreads) {  // (the same passes in every thread)
        const int n_it = min(kThreads, items - base);   // items of this pass
        const int tpi = kThreads / n_it;                 // threads per item
        const int item = threadIdx.x % n_it;
        const int sub = threadIdx.x / n_it;              // < tpi for active threads
        const bool active = sub < tpi;
        const int ih = (base + item) / D4;
        const int id = ((base + item) % D4) * 4;
        const float* src = p.ws_o + (row0 + (size_t)ih * p.P) * D + id;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c0 = 0; c0 < np; c0 += kFusedLoads * tpi) {
            float4 ov[kFusedLoads];
#pragma unroll
            for (int u = 0; u < kFusedLoads; ++u) {
                const int i = c0 + sub + u * tpi;
                ov[u] = (active && i < np)
                            ? __ldcg(reinterpret_cast<const float4*>(src + (size_t)i * D))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (base == 0 && c0 == 0) {  // (the same branch for every thread)
                __syncthreads();
                for (int h = warp; h < G; h += kWarps) {
                    float mx = -INFINITY;
                    for (int i = lane; i < np; i += 32) mx = fmaxf(mx, s_m[h * np + i]);
#pragma unroll
                    for (int mask = 16; mask > 0; mask >>= 1)
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, mask));
                    float sum = 0.f;
                    for (int i = lane; i < np; i += 32) {
                        const float l = s_w[h * np + i];
                        // l == 0: nothing attended; a NaN (bad page) is kept so it reaches the output.
                        const float w = (l == 0.f) ? 0.f : ex2(s_m[h * np + i] - mx) * l;
                        s_w[h * np + i] = w;
                        sum += w;
                    }
#pragma unroll
                    for (int mask = 16; mask > 0; mask >>= 1)
                        sum += __shfl_xor_sync(0xffffffffu, sum, mask);
                    if (lane == 0) {
                        s_M[h] = mx;
                        s_L[h] = sum;
                    }
                }
                __syncthreads();
            }
#pragma unroll
            for (int u = 0; u < kFusedLoads; ++u) {
                const int i = c0 + sub + u * tpi;
                const float w = (active && i < np) ? s_w[ih * np + i] : 0.f;
                acc.x += w * ov[u].x;
                acc.y += w * ov[u].y;
                acc.z += w * ov[u].z;
                acc.w += w * ov[u].w;
            }
        }
        if (tpi > 1) {  // (only with fewer items than threads: a single pass)
            if (active) reinterpret_cast<float4*>(scratch)[sub * n_it + item] = acc;
            __syncthreads();
            if (sub == 0) {
                for (int t = 1; t < tpi; ++t) {
                    const float4 a = reinterpret_cast<const float4*>(scratch)[t * n_it + item];
                    acc.x += a.x;
                    acc.y += a.y;
                    acc.z += a.z;
                    acc.w += a.w;
                }
            }
        }
        if (sub == 0) {
            const float lam = s_L[ih];
            const float inv = 1.f / lam;
            const size_t bh = (size_t)b * p.Hq + h0 + ih;
            store4<T>(reinterpret_cast<T*>(p.out) + bh * D + id, acc.x * inv, acc.y * inv,
                      acc.z * inv, acc.w * inv);
            if (id == 0) p.lse[bh] = (s_M[ih] + log2f(lam)) * 0.69314718055994531f;
        }
    }
}

// ---- Merge inside a thread-block cluster.  With plan.cluster = C the C
// partitions of a (sequence, KV head, head chunk) run as one cluster (grid.x =
// C, cluster C x 1 x 1).  Each CTA leaves its partial -- the normalised o of
// its G heads and their (m, l) -- in its own shared memory (the idle page
// ring), the cluster synchronises, and every CTA then merges a 1/C share of
// the (head, 4-dim column) items by reading all C partials through
// distributed shared memory (the log-sum-exp algebra of Phase 2 in the commit
// note).  No partial goes through global memory, no counter is needed, and
// there is no second launch.  A second cluster barrier keeps every CTA's
// shared memory alive until all peers have read it.  Every CTA of the cluster
// reaches both barriers (no path returns between them), and every wait before
// them is bounded.
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ int cluster_size() {
    uint32_t n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return (int)n;
}

// Shared-memory address `addr` of this CTA mapped to the same offset in CTA
// `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Layout of a CTA's partial in its shared memory (the idle page ring):
// o [G][D] (normalised), then m [G] (log2 domain) and l [G].
template <int D>
struct ClusterPartial {
    __host__ __device__ static constexpr int o_off(int h, int d) { return (h * D + d) * 4; }
    __host__ __device__ static constexpr int m_off(int G, int h) { return (G * D + h) * 4; }
    __host__ __device__ static constexpr int l_off(int G, int h) { return (G * D + G + h) * 4; }
    static constexpr int kMaxBytes = (kMaxHeadsPerCta * D + 2 * kMaxHeadsPerCta) * 4;
};

// A CTA with nothing to contribute (no page of its partition is attended,
// or a bad page id: then l = NaN, which the merge carries to the output).
// Its o stays unwritten: the merge reads no rank past the attended
// partitions, and a NaN weight makes the output NaN whatever o holds.
template <int D>
__device__ __forceinline__ void cluster_partial_fill(float* part, int G, float m, float l) {
    for (int h = threadIdx.x; h < G; h += kThreads) {
        part[ClusterPartial<D>::m_off(G, h) / 4] = m;
        part[ClusterPartial<D>::l_off(G, h) / 4] = l;
    }
}

// num_parts: the sequence's partitions that attend anything.  Cluster rank c
// serves partition c, so ranks num_parts and up have nothing to contribute
// and are not read at all.
template <int D, typename T>
__device__ __forceinline__ void cluster_merge(const AttendParams& p, int b, int h0, int G,
                                              const float* part, int num_parts) {
    __syncthreads();    // this CTA's partial is complete
    cluster_barrier();  // ... and so is every peer's
    const int C = min(cluster_size(), num_parts);  // the peers read below
    const int rank = (int)cluster_rank();
    const int per_c = cluster_size();               // every rank takes a share of the items
    const uint32_t base = smem_u32(part);
    constexpr int D4 = D / 4;
    const int items = G * D4;
    // This CTA merges a contiguous block of the (head, 4-dim column) items,
    // one thread per item, so that a warp's loads from one peer (and its
    // output stores) cover consecutive addresses.  All C partials' (m, l, o)
    // loads of an item are issued before any is used, so the merge costs one
    // distributed-shared-memory round trip.
    const int per = (items + per_c - 1) / per_c;
    const int it_end = min(items, (rank + 1) * per);
    for (int it = rank * per + (int)threadIdx.x; it < it_end; it += kThreads) {
        const int h = it / D4;
        const int d = (it % D4) * 4;
        float mv[kMaxClusterParts], lv[kMaxClusterParts];
        float4 ov[kMaxClusterParts];
#pragma unroll
        for (int c = 0; c < kMaxClusterParts; ++c) {
            if (c < C) {
                mv[c] = ld_cluster_f32(map_to_rank(base + ClusterPartial<D>::m_off(G, h), c));
                lv[c] = ld_cluster_f32(map_to_rank(base + ClusterPartial<D>::l_off(G, h), c));
                ov[c] = ld_cluster_v4(map_to_rank(base + ClusterPartial<D>::o_off(h, d), c));
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int c = 0; c < kMaxClusterParts; ++c)
            if (c < C) M = fmaxf(M, mv[c]);
        float lam = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kMaxClusterParts; ++c) {
            // l >= 1 for a partition that attends anything; NaN (a bad page
            // id, a timed-out copy) is kept.  So every value loaded above
            // is used: all of this thread's remote loads have returned
            // before its stores below, and so before the second barrier.
            if (c < C && lv[c] != 0.f) {
                const float w = ex2(mv[c] - M) * lv[c];
                lam += w;
                acc.x += w * ov[c].x;
                acc.y += w * ov[c].y;
                acc.z += w * ov[c].z;
                acc.w += w * ov[c].w;
            }
        }
        const float inv = lam == 0.f ? 0.f : 1.f / lam;  // empty context: out 0, lse -inf
        const size_t bh = (size_t)b * p.Hq + h0 + h;
        store4<T>(reinterpret_cast<T*>(p.out) + bh * D + d, acc.x * inv, acc.y * inv,
                  acc.z * inv, acc.w * inv);
        if (d == 0)
            p.lse[bh] = lam == 0.f ? -INFINITY : (M + log2f(lam)) * 0.69314718055994531f;
    }
    // Every peer is done reading this CTA's shared memory.  A relaxed arrive:
    // this CTA wrote nothing its peers read after it, and its remote loads
    // have all returned (their values feed the stores above).  The release
    // form cost about 0.3 us more per step on GB300 (Llama-3.2-1B shapes
    // 6.0 vs 5.8 us, Gemma-2 13.7 vs 13.4 us), also with the stores moved
    // behind the barrier.
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---- Rotary embedding on the tensor-core path (fp16 and bf16, head dims up
// to 128).
// The rotate-half partner of dim i (i < D/2) is dim i + D/2, which lies in
// k-step kk + KT/2 of the same mma fragment slot as dim i in k-step kk: a lane
// rotates its K fragments in registers, pairing fragment kk with kk + KT/2,
// and never writes a rotated page back.  Rotated values are fp32 split into
// a head and a remainder of the cache's type (about 22 significant bits for
// fp16, 16 for bf16), and q.K takes K_hi q_hi + K_hi q_lo + K_lo q_hi, so the
// scores keep nearly fp32 accuracy (a single fp16 rounding of the rotated q
// or K would cost ~3e-4 on the LSE).

// Packed 16-bit pairs <-> fp32 pairs, and the head + remainder split, per
// element type.
template <typename T>
struct RopeIO;

template <>
struct RopeIO<__half> {
    __device__ static __forceinline__ float2 unpack(uint32_t u) {
        return __half22float2(*reinterpret_cast<__half2*>(&u));
    }
    // v = hi + lo with hi = fp16(v) and lo = fp16(v - hi), elementwise.
    __device__ static __forceinline__ void split(float2 v, uint32_t& hi, uint32_t& lo) {
        __half2 h = __float22half2_rn(v);
        const float2 hb = __half22float2(h);
        __half2 l = __float22half2_rn(make_float2(v.x - hb.x, v.y - hb.y));
        hi = *reinterpret_cast<uint32_t*>(&h);
        lo = *reinterpret_cast<uint32_t*>(&l);
    }
};

template <>
struct RopeIO<__nv_bfloat16> {
    __device__ static __forceinline__ float2 unpack(uint32_t u) {
        return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u));
    }
    // v = hi + lo with hi = bf16(v) and lo = bf16(v - hi): about 16 significant bits.
    __device__ static __forceinline__ void split(float2 v, uint32_t& hi, uint32_t& lo) {
        __nv_bfloat162 h = __float22bfloat162_rn(v);
        const float2 hb = __bfloat1622float2(h);
        __nv_bfloat162 l = __float22bfloat162_rn(make_float2(v.x - hb.x, v.y - hb.y));
        hi = *reinterpret_cast<uint32_t*>(&h);
        lo = *reinterpret_cast<uint32_t*>(&l);
    }
};

// x = dims (i, i + 1) of the first half, y = their partners (i + D/2,
// i + D/2 + 1), as packed 16-bit pairs; (c, s) = cos, sin of their angles.
// The rotated pair x' = x c - y s, y' = y c + x s, split into head + rest.
template <typename T>
__device__ __forceinline__ void rope_rot_split(uint32_t x16, uint32_t y16, float2 c, float2 s,
                                               uint32_t& xh, uint32_t& xl, uint32_t& yh,
                                               uint32_t& yl) {
    const float2 x = RopeIO<T>::unpack(x16);
    const float2 y = RopeIO<T>::unpack(y16);
    const float2 xr = __ffma2_rn(x, c, __fmul2_rn(y, make_float2(-s.x, -s.y)));
    const float2 yr = __ffma2_rn(y, c, __fmul2_rn(x, s));
    RopeIO<T>::split(xr, xh, xl);
    RopeIO<T>::split(yr, yh, yl);
}

// (c, s) <- (c, s) turned by the angles whose cos/sin are t = (cos f, sin f,
// cos f+1, sin f+1): c' = c cr - s sr, s' = s cr + c sr, per element.
__device__ __forceinline__ void rope_turn_pair(float2& c, float2& s, float4 t) {
    const float2 cr = make_float2(t.x, t.z), sr = make_float2(t.y, t.w);
    const float2 cn = __ffma2_rn(c, cr, __fmul2_rn(s, make_float2(-sr.x, -sr.y)));
    const float2 sn = __ffma2_rn(s, cr, __fmul2_rn(c, sr));
    c = cn;
    s = sn;
}

// Before the dependency wait of a programmatic dependent launch, per warp:
// read the sequence length and this warp's first page ids (relative pages
// first, first + step, ... below limit) as hints and request its first
// prewait_prefetch pages (K and V) into L2, so that they
// stream in while the previous grid drains.  The values read here may be
// stale (the previous grid may still be writing them): they are only
// bounds-checked prefetch addresses, and everything is read again after the
// wait, so a stale hint costs one useless prefetch.  L2-only loads, so that
// nothing read here sits in L1 afterwards.
__device__ __forceinline__ void prefetch_first_pages(const AttendParams& p, int part0, int kvh,
                                                     int b, int pp, int first, int step,
                                                     int limit, int lane, int D) {
    int Lh = 0;
    if (lane == 0) Lh = __ldcg(p.context_lens + b);
    Lh = __shfl_sync(0xffffffffu, Lh, 0);
    const SeqSpan sp = seq_span(Lh, p.window, p.max_ctx, p.maxp, pp);
    if (!sp.valid || part0 >= sp.num_parts) return;
    const int pgA = sp.first_page + part0 * pp;
    const int n_range = min(p.parts_per_cta * pp, sp.end_page - pgA);
    const int j = first + step * lane;  // this lane: page `lane` of the warp
    if (lane < p.prewait_prefetch && j < min(n_range, limit)) {
        const int id = __ldcg(p.block_tables + (size_t)b * p.maxp + pgA + j);
        if (id >= 0 && id < p.num_pages) {
            const size_t off = ((size_t)id * p.Hkv + kvh) * (size_t)(kPageSize * D);
            prefetch_l2(p.k + off, kPageSize * D * 2);
            prefetch_l2(p.v + off, kPageSize * D * 2);
        }
    }
}

// Work-balanced partitions (plan.balanced = X > 0): the X CTAs along grid.x
// of a (KV head, head chunk) share the whole batch, so that a long sequence
// gets more CTAs than a short one.  With pp from balanced_pp, sequence b gets
// n_b = max(1, ceil(pages_b / pp)) consecutive CTAs, in batch order.  Every
// CTA computes this map from the same B lengths (one load per thread, B <=
// kThreads) and takes the (sequence, partition) item its x falls in; with
// x >= sum_b n_b it has none.  `hint`: lengths read with L2-only loads, for
// the prefetch addresses before the dependency wait (they may be stale).
struct BalancedItem {
    int b, part, pp;
};

__device__ __forceinline__ bool balanced_item(const AttendParams& p, int x, bool hint,
                                              BalancedItem& it) {
    __shared__ int s_red[kWarps];
    __shared__ int s_item[2];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int B = p.B, X = p.balanced;
    int pages = 0;
    if (t < B) {
        const int L = hint ? __ldcg(p.context_lens + t) : p.context_lens[t];
        pages = balanced_seq_pages(L, p.window, p.max_ctx, p.maxp);
    }
    if (t == 0) s_item[0] = -1;
    const int pp = balanced_pp(pages, B, X, s_red);
    const int n = t < B ? max(1, (pages + pp - 1) / pp) : 0;
    int inc = n;  // inclusive scan of n over the CTA
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, m);
        if (lane >= m) inc += o;
    }
    __syncthreads();  // every read of s_red above is done
    if (lane == 31) s_red[warp] = inc;
    __syncthreads();
    for (int w = 0; w < warp; ++w) inc += s_red[w];
    const int exc = inc - n;
    if (t < B && x >= exc && x < inc) {
        s_item[0] = t;
        s_item[1] = x - exc;
    }
    __syncthreads();
    it.b = s_item[0];
    it.part = s_item[1];
    it.pp = pp;
    __syncthreads();  // s_item and s_red may be reused by a second call
    return it.b >= 0;
}

static_assert(ClusterPartial<64>::kMaxBytes <= MmaCfg<64>::kWideXOff &&
                  ClusterPartial<96>::kMaxBytes <= MmaCfg<96>::kWideXOff &&
                  ClusterPartial<128>::kMaxBytes <= MmaCfg<128>::kWideXOff &&
                  ClusterPartial<256>::kMaxBytes <= MmaCfg<256>::kWideXOff,
              "the cluster partial sits in the ring in front of the one-round combine");

// SPLIT: partials for a merge (else the final rows).  CLUSTER (with SPLIT):
// the partitions of a group form one cluster and merge in it; a separate
// instance, so that the other instances carry none of its code.  ROPE: q and
// each K row are rotated to their positions before q.K.
template <int D, typename T, bool SPLIT, bool CLUSTER, bool ROPE, bool DEEP = false>
__global__ void __launch_bounds__(kThreads, MmaCfg<D, ROPE, DEEP>::kMinBlocks)
    attend_mma_kernel(const AttendParams p, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV) {
    using Cfg = MmaCfg<D, ROPE, DEEP>;
    constexpr int NS = Cfg::kStages;
    constexpr int PB = Cfg::kPageBytes;
    constexpr int KT = D / 16;  // k-steps of q.K, m-tiles of P.V

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;  // 128-byte swizzle needs 1 KiB alignment
    unsigned char* base = smem_raw + (base_u32 - raw_u32);
    unsigned char* ring = base;
    float* xbuf = reinterpret_cast<float*>(base + Cfg::kRingBytes);  // last-CTA merge scratch
    // The CTA's page ids (up to kMaxStagedPages) live in the merge scratch:
    // they are read only while pages stream, the merge runs after the last page.
    int* s_pid = reinterpret_cast<int*>(xbuf);
    float* s_ml = reinterpret_cast<float*>(base + Cfg::kRingBytes + Cfg::kXBytes);  // [warps][m|l|n][8]
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_ml + kWarps * kMaxHeadsPerCta * 3);
    // rotary tables (ROPE): (cos, sin) per frequency of the 8-token turn and of
    // the turn by one step of a warp's pages (16 * wpp tokens; "r64")
    float2* s_r8 = reinterpret_cast<float2*>(bars + kWarps * NS);
    float2* s_r64 = s_r8 + D / 2;
    __shared__ int s_flag;

    const int G = p.heads_per_cta;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ppc = p.parts_per_cta;
    const int kvh = blockIdx.y / p.nchunk;
    const int h0 = kvh * p.g + (blockIdx.y % p.nchunk) * G;
    // This CTA's sequence, first partition, partition size in pages and
    // partial row.  A work-balanced plan (p.balanced) decides them on the
    // device from the batch's lengths (balanced_item): first from hints for
    // the prefetch, then for real after the dependency wait.
    int b = blockIdx.z;
    int part0 = blockIdx.x * ppc;
    int pp = p.pages_per_part;
    int slot = blockIdx.x;
    const int wpp = kWarps / ppc;  // warps per partition (ppc is 1, 2 or 4)
    const int wq = warp / wpp;     // this warp's partition slot within the CTA
    const int wl = warp % wpp;     // and its place among that partition's warps
    // relative page of this warp's i-th page, and its page count in a range
    // of n_range pages
    auto wpage = [&](int i) { return wq * pp + wl + i * wpp; };
    auto warp_pages = [&](int n_range) {
        const int q_end = min((wq + 1) * pp, n_range);
        const int first = wq * pp + wl;
        return q_end > first ? (q_end - first + wpp - 1) / wpp : 0;
    };
    const uint32_t bar_w = smem_u32(bars) + warp * NS * 8;
    const uint32_t ring_w = smem_u32(ring) + warp * NS * PB;

    // Ring copy of item `item` (K0, V0, K1, V1, ... of this warp's pages) from
    // page `id` of the pool.
    auto issue_page = [&](int item, int id) {
        const int slot = item % NS;
        const CUtensorMap* map = (item & 1) ? &tmV : &tmK;
        const int y = (id * p.Hkv + kvh) * kPageSize;
        const uint32_t bar = bar_w + slot * 8;
        // (stall_tx, a test hook, is 0 outside tests)
        mbar_arrive_expect_tx(bar, PB + (item == 0 ? p.stall_tx : 0));
        if constexpr (Cfg::kRows64) {
            tma_load_3d(ring_w + slot * PB, map, 0, 0, y, bar);
        } else {
            tma_load_3d(ring_w + slot * PB, map, 0, y, 0, bar);  // the whole page, all slabs
        }
    };

    // Programmatic dependent launch: let the merge grid (or the next call's
    // grid) be scheduled now, and read nothing before the grid this one
    // depends on has completed -- except the prefetch hints.
    allow_dependent_launch();
    if (threadIdx.x == 0) {
        s_flag = 0;
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmK)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmV)) : "memory");
    }
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < NS; ++s) mbar_init(bar_w + s * 8, 1);
        fence_mbar_init();
    }
    // Work-balanced plans: split instances without a cluster or rotary
    // embedding (the run-time sequence and partition cost the D = 256 rotary
    // instances, already at 255 registers, a spill).
    constexpr bool kBalancedInstance = SPLIT && !CLUSTER && !ROPE;
    if (p.prewait_prefetch) {
        BalancedItem hi{b, part0, pp};
        if (!(kBalancedInstance && p.balanced) || balanced_item(p, blockIdx.x, true, hi))
            prefetch_first_pages(p, hi.part, kvh, hi.b, hi.pp, wq * hi.pp + wl, wpp,
                                 (wq + 1) * hi.pp, lane, D);
    }
    if constexpr (ROPE) {
        // (kernel parameters only: no input is read)
        for (int f = threadIdx.x; f < D / 2; f += kThreads) {
            float c, sn;
            rope_twiddle(8, p.rope_phi[0][f], p.rope_phi[1][f], c, sn);
            s_r8[f] = make_float2(c, sn);
            rope_twiddle(wpp * kPageSize, p.rope_phi[0][f], p.rope_phi[1][f], c, sn);
            s_r64[f] = make_float2(c, sn);
        }
    }
    // Page ids read together with the length (instances without rotary
    // embedding, fixed partitions): the length read before the dependency
    // wait, as a hint, says which block-table entries this CTA will most
    // likely stage -- its range plus one page either side.  Those entries
    // are loaded after the wait, in the same round trip as the length
    // itself, and used only if the length's real range lies inside them
    // (otherwise they are loaded again).  A decode step moves the range by at
    // most a page, so this saves one dependent memory round trip per CTA.
    constexpr bool kSpecIds = !ROPE;
    constexpr int kSpecLoads = 3;  // per thread: ranges of up to 3 * kThreads entries
    const bool spec_ids = kSpecIds && !(kBalancedInstance && p.balanced);
    int len_hint = 0;
    if (spec_ids) len_hint = __ldcg(p.context_lens + b);
    __syncthreads();  // barriers and rotary tables initialised
    wait_for_prerequisite_grid();
    if (kBalancedInstance && p.balanced) {
        BalancedItem it;
        const bool has_item = balanced_item(p, blockIdx.x, false, it);
        // (every CTA finds the same partition size; one leaves it for the merge kernel)
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *p.ws_info = it.pp;
        if (!has_item) return;  // more CTAs than items
        b = it.b;
        part0 = it.part;  // (one partition per CTA)
        pp = it.pp;
        slot = it.part;
    }

    const int len = p.context_lens[b];
    int spec_lo = 0, spec_n = 0;  // block-table entries [spec_lo, spec_lo + spec_n) of row b
    int spec[kSpecIds ? kSpecLoads : 1];
    if (spec_ids) {
        const SeqSpan hs = seq_span(len_hint, p.window, p.max_ctx, p.maxp, pp);
        if (hs.valid && part0 < hs.num_parts) {
            const int a = hs.first_page + part0 * pp;
            const int n = min(ppc * pp, hs.end_page - a);
            spec_lo = max(0, a - 1);
            spec_n = min(p.maxp, a + n + 1) - spec_lo;
            if (spec_n > kSpecLoads * kThreads) spec_n = 0;
        }
#pragma unroll
        for (int u = 0; u < (kSpecIds ? kSpecLoads : 1); ++u) {
            const int j = u * kThreads + (int)threadIdx.x;
            spec[u] = j < spec_n ? p.block_tables[(size_t)b * p.maxp + spec_lo + j] : 0;
        }
    }
    const SeqSpan sp = seq_span(len, p.window, p.max_ctx, p.maxp, pp);
    T* const out = reinterpret_cast<T*>(p.out);
    auto fill_rows = [&](int slot, float o_val, float m_val, float l_val, float lse_val) {
        for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
            const int h = idx / D, d = idx % D;
            const size_t bh = (size_t)b * p.Hq + h0 + h;
            if constexpr (SPLIT) {
                const size_t row = bh * p.P + slot;  // (the CTA's partial row)
                p.ws_o[row * D + d] = o_val;
                if (d == 0) {
                    p.ws_m[row] = m_val;
                    p.ws_l[row] = l_val;
                }
            } else {
                out[bh * D + d] = Elem<T>::from_float(o_val);
                if (d == 0) p.lse[bh] = lse_val;
            }
        }
    };
    const bool fused = SPLIT && !CLUSTER && p.merge_in_kernel;
    // Final rows written without any partial (used when nothing is merged).
    auto final_rows = [&](float o_val, float lse_val) {
        for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
            const int h = idx / D, d = idx % D;
            const size_t bh = (size_t)b * p.Hq + h0 + h;
            out[bh * D + d] = Elem<T>::from_float(o_val);
            if (d == 0) p.lse[bh] = lse_val;
        }
    };
    constexpr bool clustered = SPLIT && CLUSTER;
    float* const cpart = reinterpret_cast<float*>(ring);  // this CTA's partial (cluster merge)
    if (!sp.valid) {
        // (the same for every CTA of a cluster: they all leave here)
        if (threadIdx.x == 0 && part0 == 0 && blockIdx.y == 0) atomicOr(p.err, PA_DEVERR_BAD_LENGTH);
        if (!SPLIT || ((fused || clustered) && slot == 0)) final_rows(NAN, NAN);
        return;  // with a separate merge, the merge writes the NaN rows
    }
    if (part0 >= sp.num_parts) {
        // Nothing attended here.  The group's rows are written here only for
        // an empty context (out = 0, lse = -inf) when no merge kernel runs.
        if (clustered) {
            cluster_partial_fill<D>(cpart, G, -INFINITY, 0.f);
            cluster_merge<D, T>(p, b, h0, G, cpart, sp.num_parts);
            return;
        }
        if (!SPLIT || (fused && sp.num_parts == 0 && slot == 0)) final_rows(0.f, -INFINITY);
        return;
    }
    const int nparts = min(ppc, sp.num_parts - part0);
    const int pgA = sp.first_page + part0 * pp;           // first page of this CTA
    const int n_range = min(nparts * pp, sp.end_page - pgA);  // pages of this CTA

    // Stage the CTA's page ids, each checked before any copy (a bad id is
    // never read through): from the entries loaded with the length when
    // they cover the range, else loaded now.
    if (spec_ids && spec_n > 0 && pgA >= spec_lo && pgA + n_range <= spec_lo + spec_n) {
        const int shift = pgA - spec_lo;
#pragma unroll
        for (int u = 0; u < (kSpecIds ? kSpecLoads : 1); ++u) {
            const int j = u * kThreads + (int)threadIdx.x - shift;
            if (j >= 0 && j < n_range) {
                int id = spec[u];
                if (id < 0 || id >= p.num_pages) {
                    s_flag = 1;
                    id = 0;
                }
                s_pid[j] = id;
            }
        }
    } else {
        for (int j = threadIdx.x; j < n_range; j += kThreads) {
            int id = p.block_tables[(size_t)b * p.maxp + pgA + j];
            if (id < 0 || id >= p.num_pages) {
                s_flag = 1;
                id = 0;
            }
            s_pid[j] = id;
        }
    }
    __syncthreads();
    if (s_flag) {
        if (threadIdx.x == 0) atomicOr(p.err, PA_DEVERR_BAD_PAGE);
        if (clustered) {  // no copy has been issued: the ring is free
            cluster_partial_fill<D>(cpart, G, NAN, NAN);
            cluster_merge<D, T>(p, b, h0, G, cpart, sp.num_parts);
            return;
        }
        fill_rows(slot, NAN, NAN, NAN, NAN);
        if (fused) group_arrive_and_merge<D, T>(p, sp, b, h0, G, xbuf, s_ml,
                                                reinterpret_cast<float*>(ring));
        return;
    }

    // ---- this warp's pages: the CTA's ppc partitions each get kWarps / ppc
    // warps (wpp), and warp wl of partition slot wq streams the partition's
    // pages wl, wl + wpp, ... (relative page j = wq * pp + wl + i * wpp);
    // items K0, V0, K1, V1, ...
    const int nk = warp_pages(n_range);
    const int n_items = 2 * nk;
    auto issue = [&](int item) { issue_page(item, s_pid[wpage(item >> 1)]); };
    if (lane == 0) {
        for (int i = 0; i < NS && i < n_items; ++i) issue(i);
    }
    int issued = min(NS, n_items);
    bool ok = true;

    // q as the B operand of q.K: lane holds q[head = lane/4][dims kk*16 + (lane%4)*2 + {0,1}, +8]
    const int qh = lane >> 2;
    const bool q_ok = qh < G;
    uint32_t qb[KT][2];
    {
        const __half* qrow = p.q + ((size_t)b * p.Hq + h0 + (q_ok ? qh : 0)) * D + (lane & 3) * 2;
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
            qb[kk][0] = q_ok ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16) : 0u;
            qb[kk][1] = q_ok ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8) : 0u;
        }
    }
    // Rotary instances: q rotated to position L - 1, as fp16 head (qb) + rest
    // (ql).  Slot r of k-step kk holds dims kk*16 + (lane%4)*2 + r*8 + {0, 1};
    // their partners sit in the same slot of k-step kk + KT/2.
    uint32_t ql[ROPE ? KT : 1][2];
    if constexpr (ROPE) {
        const int qpos = sp.L - 1;
#pragma unroll
        for (int kk = 0; kk < KT / 2; ++kk) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int f = kk * 16 + (lane & 3) * 2 + r * 8;
                float c0, s0, c1, s1;
                rope_twiddle(qpos, p.rope_phi[0][f], p.rope_phi[1][f], c0, s0);
                rope_twiddle(qpos, p.rope_phi[0][f + 1], p.rope_phi[1][f + 1], c1, s1);
                rope_rot_split<T>(qb[kk][r], qb[kk + KT / 2][r], make_float2(c0, c1),
                               make_float2(s0, s1), qb[kk][r], ql[kk][r], qb[kk + KT / 2][r],
                               ql[kk + KT / 2][r]);
            }
        }
    }
    // Rotary state (ROPE): cos/sin of this lane's frequencies at its first
    // token row of the current page, slot i = kk*2 + r <-> frequencies
    // kk*16 + (lane%4)*2 + r*8 + {0, 1}.  Evaluated exactly on every 32nd
    // page of the warp and turned by one step of the warp's pages (wpp pages,
    // the s_r64 table) in between: 31 turns add a few 1e-6 of relative error to the angles'
    // cos/sin, far below what the scores can show, and the exact evaluations
    // (32 per lane) are the costliest part of a page.
    float2 rc[ROPE ? KT : 1], rs[ROPE ? KT : 1];

    const int tok0 = lane >> 2;  // this lane's tokens of a page: tok0 and tok0 + 8
    const int hA = (lane & 3) * 2;  // and its heads hA, hA + 1
    // ldmatrix row/chunk roles of this lane
    const int ld_j = lane >> 3;
    const int ld_i = lane & 7;
    const int k_row = ld_i + (ld_j & 1) * 8;  // q.K: matrices (rows 0-7|8-15) x (chunk +0|+1)
    const int k_chk = ld_j >> 1;
    const int v_row = ld_i + (ld_j >> 1) * 8; // P.V (trans): (chunk +0|+1) x (tokens 0-7|8-15)
    const int v_chk = ld_j & 1;
    int consumed = 0;
    int k = 0;  // this warp's next page (index into its stream)

    {
        float o[KT][4];
#pragma unroll
        for (int mt = 0; mt < KT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        float m_run[2] = {-INFINITY, -INFINITY};
        float l_run[2] = {0.f, 0.f};   // exp-sum of the fp32 weights
        float n_run[2] = {0.f, 0.f};   // exp-sum of the fp16-rounded weights

        for (; ok && k < nk; ++k) {
            const int page_pos = (pgA + wpage(k)) * kPageSize;
            // ---------------- K page: S^T = K . Q^T
            {
                const int item = 2 * k;
                const bool got = mbar_wait_bounded(bar_w + (item % NS) * 8, (item / NS) & 1);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                consumed = item + 1;
            }
            const uint32_t kaddr = ring_w + ((2 * k) % NS) * PB;
            float ca[4] = {0.f, 0.f, 0.f, 0.f}, cb[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (ROPE) {
                // the rotary state at this page's row tok0 (rc, rs); row tok0 + 8
                // is derived per k-step below, for the two slots it uses
#pragma unroll
                for (int i = 0; i < KT; ++i) {
                    const int f = (i >> 1) * 16 + (lane & 3) * 2 + (i & 1) * 8;
                    if ((k & 31) == 0) {
                        float c0, s0, c1, s1;
                        rope_twiddle(page_pos + tok0, p.rope_phi[0][f], p.rope_phi[1][f], c0, s0);
                        rope_twiddle(page_pos + tok0, p.rope_phi[0][f + 1], p.rope_phi[1][f + 1],
                                     c1, s1);
                        rc[i] = make_float2(c0, c1);
                        rs[i] = make_float2(s0, s1);
                    } else {
                        rope_turn_pair(rc[i], rs[i], *reinterpret_cast<const float4*>(s_r64 + f));
                    }
                }
#pragma unroll
                for (int kk = 0; kk < KT / 2; ++kk) {
                    // fragments: a0/a2 row tok0, a1/a3 row tok0 + 8; a0/a1 slot r = 0, a2/a3 r = 1
                    const int f0 = kk * 16 + (lane & 3) * 2;
                    float2 c8a = rc[2 * kk], s8a = rs[2 * kk];
                    float2 c8b = rc[2 * kk + 1], s8b = rs[2 * kk + 1];
                    rope_turn_pair(c8a, s8a, *reinterpret_cast<const float4*>(s_r8 + f0));
                    rope_turn_pair(c8b, s8b, *reinterpret_cast<const float4*>(s_r8 + f0 + 8));
                    uint32_t x[4], y[4], xh[4], xl[4], yh[4], yl[4];
                    ldsm_x4(kaddr + swz<D>(k_row, kk * 2 + k_chk), x[0], x[1], x[2], x[3]);
                    ldsm_x4(kaddr + swz<D>(k_row, (kk + KT / 2) * 2 + k_chk), y[0], y[1], y[2],
                            y[3]);
                    rope_rot_split<T>(x[0], y[0], rc[2 * kk], rs[2 * kk], xh[0], xl[0], yh[0], yl[0]);
                    rope_rot_split<T>(x[1], y[1], c8a, s8a, xh[1], xl[1], yh[1], yl[1]);
                    rope_rot_split<T>(x[2], y[2], rc[2 * kk + 1], rs[2 * kk + 1], xh[2], xl[2], yh[2],
                                      yl[2]);
                    rope_rot_split<T>(x[3], y[3], c8b, s8b, xh[3], xl[3], yh[3], yl[3]);
                    const int k2 = kk + KT / 2;
                    Elem<T>::mma(ca, xh[0], xh[1], xh[2], xh[3], qb[kk][0], qb[kk][1]);
                    Elem<T>::mma(ca, xh[0], xh[1], xh[2], xh[3], ql[kk][0], ql[kk][1]);
                    Elem<T>::mma(ca, xl[0], xl[1], xl[2], xl[3], qb[kk][0], qb[kk][1]);
                    Elem<T>::mma(cb, yh[0], yh[1], yh[2], yh[3], qb[k2][0], qb[k2][1]);
                    Elem<T>::mma(cb, yh[0], yh[1], yh[2], yh[3], ql[k2][0], ql[k2][1]);
                    Elem<T>::mma(cb, yl[0], yl[1], yl[2], yl[3], qb[k2][0], qb[k2][1]);
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < KT; ++kk) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(kaddr + swz<D>(k_row, kk * 2 + k_chk), a0, a1, a2, a3);
                    if (kk & 1)
                        Elem<T>::mma(cb, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
                    else
                        Elem<T>::mma(ca, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
                }
            }
            __syncwarp();
            if (lane == 0 && 2 * k + NS < n_items) {
                fence_proxy_async_smem();
                issue(2 * k + NS);
            }
            if (2 * k + NS < n_items) issued = 2 * k + NS + 1;

            // ---------------- online softmax (log2 domain); lane: tokens tok0, tok0+8; heads hA, hA+1
            const bool v0 = page_pos + tok0 >= sp.start && page_pos + tok0 < sp.L;
            const bool v1 = page_pos + tok0 + 8 >= sp.start && page_pos + tok0 + 8 < sp.L;
            float s00 = v0 ? (ca[0] + cb[0]) * p.scale_log2 : -INFINITY;  // token0, head A
            float s01 = v0 ? (ca[1] + cb[1]) * p.scale_log2 : -INFINITY;  // token0, head B
            float s10 = v1 ? (ca[2] + cb[2]) * p.scale_log2 : -INFINITY;  // token1, head A
            float s11 = v1 ? (ca[3] + cb[3]) * p.scale_log2 : -INFINITY;  // token1, head B
            float mA = fmaxf(s00, s10), mB = fmaxf(s01, s11);
#pragma unroll
            for (int mask = 4; mask < 32; mask <<= 1) {
                mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, mask));
                mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, mask));
            }
            if (__any_sync(0xffffffffu, mA > m_run[0] || mB > m_run[1])) {
                const float nA = fmaxf(m_run[0], mA), nB = fmaxf(m_run[1], mB);
                const float aA = (nA == -INFINITY) ? 1.f : ex2(m_run[0] - nA);
                const float aB = (nB == -INFINITY) ? 1.f : ex2(m_run[1] - nB);
                m_run[0] = nA;
                m_run[1] = nB;
                l_run[0] *= aA;
                l_run[1] *= aB;
                n_run[0] *= aA;
                n_run[1] *= aB;
#pragma unroll
                for (int mt = 0; mt < KT; ++mt) {
                    o[mt][0] *= aA;
                    o[mt][2] *= aA;
                    o[mt][1] *= aB;
                    o[mt][3] *= aB;
                }
            }
            const float p00 = (s00 == -INFINITY) ? 0.f : ex2(s00 - m_run[0]);
            const float p01 = (s01 == -INFINITY) ? 0.f : ex2(s01 - m_run[1]);
            const float p10 = (s10 == -INFINITY) ? 0.f : ex2(s10 - m_run[0]);
            const float p11 = (s11 == -INFINITY) ? 0.f : ex2(s11 - m_run[1]);
            float r00, r01, r10, r11;
            const uint32_t top = Elem<T>::pack2(p00, p01, r00, r01);  // P[tok0][hA, hB]
            const uint32_t bot = Elem<T>::pack2(p10, p11, r10, r11);  // P[tok0 + 8][hA, hB]
            l_run[0] += p00 + p10;
            l_run[1] += p01 + p11;
            // P^T fragments: lane gets P[tokens (lane%4)*2 + {0,1} (+8)][head lane/4]
            const uint32_t pb0 = movmatrix_trans(top);
            const uint32_t pb1 = movmatrix_trans(bot);
            uint32_t pc0 = 0u, pc1 = 0u;  // bf16 only: the remainders P - head
            if constexpr (std::is_same<T, __nv_bfloat16>::value) {
                float e00, e01, e10, e11;
                const uint32_t ltop = Elem<T>::pack2(p00 - r00, p01 - r01, e00, e01);
                const uint32_t lbot = Elem<T>::pack2(p10 - r10, p11 - r11, e10, e11);
                r00 += e00;
                r01 += e01;
                r10 += e10;
                r11 += e11;
                pc0 = movmatrix_trans(ltop);
                pc1 = movmatrix_trans(lbot);
            }
            n_run[0] += r00 + r10;
            n_run[1] += r01 + r11;

            // ---------------- V page: O^T += V^T . P^T
            {
                const int item = 2 * k + 1;
                const bool got = mbar_wait_bounded(bar_w + (item % NS) * 8, (item / NS) & 1);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                consumed = item + 1;
            }
            const uint32_t vaddr = ring_w + ((2 * k + 1) % NS) * PB;
            if (page_pos < sp.start || page_pos + kPageSize > sp.L) {
                // Boundary page: zero the V rows of tokens outside [start, L) so
                // that whatever those slots hold (never-written cache slots may
                // hold NaN) cannot reach the output through a zero weight.
                unsigned char* vgen = ring + warp * NS * PB + ((2 * k + 1) % NS) * PB;
                for (int idx = lane; idx < kPageSize * (D / 8); idx += 32) {
                    const int row = idx / (D / 8);
                    const int pos = page_pos + row;
                    if (pos < sp.start || pos >= sp.L)
                        *reinterpret_cast<uint4*>(vgen + swz<D>(row, idx % (D / 8))) =
                            make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
#pragma unroll
            for (int mt = 0; mt < KT; ++mt) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(vaddr + swz<D>(v_row, mt * 2 + v_chk), a0, a1, a2, a3);
                Elem<T>::mma(o[mt], a0, a1, a2, a3, pb0, pb1);
                if constexpr (std::is_same<T, __nv_bfloat16>::value)
                    Elem<T>::mma(o[mt], a0, a1, a2, a3, pc0, pc1);
            }
            __syncwarp();
            if (lane == 0 && 2 * k + 1 + NS < n_items) {
                fence_proxy_async_smem();
                issue(2 * k + 1 + NS);
            }
            if (2 * k + 1 + NS < n_items) issued = 2 * k + 1 + NS + 1;
        }
        if (!ok) {
            if (lane == 0) {
                atomicOr(p.err, PA_DEVERR_TIMEOUT);
                s_flag = 1;
            }
            // Give every copy this warp issued a bounded chance to land, so
            // that none writes into shared memory after the CTA exits or
            // while the ring holds the cluster partial.
            for (int item = consumed; item < issued; ++item)
                (void)mbar_wait_bounded(bar_w + (item % NS) * 8, (item / NS) & 1);
            consumed = issued;
        }

        // ---- combine the warp states of each of the CTA's partitions (wpp
        // warps each).  Exp-sums: lanes with equal lane%4 hold the same heads
        // over different tokens.
#pragma unroll
        for (int mask = 4; mask < 32; mask <<= 1) {
            l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], mask);
            l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], mask);
            n_run[0] += __shfl_xor_sync(0xffffffffu, n_run[0], mask);
            n_run[1] += __shfl_xor_sync(0xffffffffu, n_run[1], mask);
        }
        if (lane < 4) {
            float* ml = s_ml + warp * 3 * kMaxHeadsPerCta;
            if (hA < G) {
                ml[hA] = m_run[0];
                ml[kMaxHeadsPerCta + hA] = l_run[0];
                ml[2 * kMaxHeadsPerCta + hA] = n_run[0];
            }
            if (hA + 1 < G) {
                ml[hA + 1] = m_run[1];
                ml[kMaxHeadsPerCta + hA + 1] = l_run[1];
                ml[2 * kMaxHeadsPerCta + hA + 1] = n_run[1];
            }
        }
        constexpr int D4 = D / 4;
        // Every warp is past its last page, so the page ring is idle: all D
        // dims of every warp state go there at once (behind the cluster
        // partial) and one round combines them, with the merge's log-sum-exp
        // algebra, into the CTA's one partial (its ppc partitions together)
        // or into the final rows.
        __syncthreads();
        float* xw = reinterpret_cast<float*>(ring + Cfg::kWideXOff);
        constexpr int XS = Cfg::kWideXStride;
#pragma unroll
        for (int mt = 0; mt < KT; ++mt) {
            const int d = mt * 16 + (lane >> 2);
            if (hA < G) {
                xw[(warp * G + hA) * XS + d] = o[mt][0];
                xw[(warp * G + hA) * XS + d + 8] = o[mt][2];
            }
            if (hA + 1 < G) {
                xw[(warp * G + hA + 1) * XS + d] = o[mt][1];
                xw[(warp * G + hA + 1) * XS + d + 8] = o[mt][3];
            }
        }
        __syncthreads();
        const bool failed = s_flag != 0;
        for (int idx = threadIdx.x; idx < G * D4; idx += kThreads) {
            const int h = idx / D4;
            const int d = (idx % D4) * 4;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_ml[w * 3 * kMaxHeadsPerCta + h]);
            float Ls = 0.f, Ns = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float* ml = s_ml + w * 3 * kMaxHeadsPerCta;
                const float mw = ml[h];
                const float c = (mw == -INFINITY) ? 0.f : ex2(mw - M);
                Ls += c * ml[kMaxHeadsPerCta + h];
                Ns += c * ml[2 * kMaxHeadsPerCta + h];
                const float4 ow = *reinterpret_cast<const float4*>(xw + (w * G + h) * XS + d);
                acc.x += c * ow.x;
                acc.y += c * ow.y;
                acc.z += c * ow.z;
                acc.w += c * ow.w;
            }
            float inv = Ns > 0.f ? 1.f / Ns : 0.f;
            if (failed) {
                inv = NAN;
                M = NAN;
                Ls = NAN;
            }
            const size_t bh = (size_t)b * p.Hq + h0 + h;
            if constexpr (SPLIT) {
                const float4 ov = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
                if (clustered) {
                    *reinterpret_cast<float4*>(cpart + ClusterPartial<D>::o_off(h, d) / 4) = ov;
                    if (d == 0) {
                        cpart[ClusterPartial<D>::m_off(G, h) / 4] = M;
                        cpart[ClusterPartial<D>::l_off(G, h) / 4] = Ls;
                    }
                } else {
                    const size_t row = bh * p.P + slot;
                    *reinterpret_cast<float4*>(p.ws_o + row * D + d) = ov;
                    if (d == 0) {
                        p.ws_m[row] = M;
                        p.ws_l[row] = Ls;
                    }
                }
            } else {
                store4<T>(out + bh * D + d, acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
                if (d == 0)
                    p.lse[bh] = failed ? NAN
                                       : (Ls > 0.f ? M * 0.69314718055994531f + logf(Ls)
                                                   : -INFINITY);
            }
        }
        __syncthreads();  // the ring and s_ml are reused by the merges below
    }

    if (clustered) {
        cluster_merge<D, T>(p, b, h0, G, cpart, sp.num_parts);
        return;
    }
    if (fused) group_arrive_and_merge<D, T>(p, sp, b, h0, G, xbuf, s_ml,
                                            reinterpret_cast<float*>(ring));
}

// Whether (D, ROPE) has a deep-ring cluster instance (MmaCfg DEEP).
template <int D, bool ROPE>
constexpr bool kHasDeep = !ROPE && (D == 96 || D == 128 || D == 256);

template <int D, typename T, bool ROPE>
cudaError_t launch_attend_mma_dr(bool split, const AttendParams& p, const CUtensorMap* maps,
                                 dim3 grid, cudaStream_t stream) {
    const bool clustered = split && p.cluster > 1;
    const bool deep = clustered && p.deep && kHasDeep<D, ROPE>;
    const void* fn =
        !split ? reinterpret_cast<const void*>(&attend_mma_kernel<D, T, false, false, ROPE>)
        : clustered ? reinterpret_cast<const void*>(&attend_mma_kernel<D, T, true, true, ROPE>)
                    : reinterpret_cast<const void*>(&attend_mma_kernel<D, T, true, false, ROPE>);
    int smem = MmaCfg<D, ROPE>::kSmemBytes;
    if constexpr (kHasDeep<D, ROPE>) {
        if (deep) {
            fn = reinterpret_cast<const void*>(&attend_mma_kernel<D, T, true, true, ROPE, true>);
            smem = MmaCfg<D, ROPE, true>::kSmemBytes;
        }
    }
    constexpr int kMaxDevices = 64;
    static std::atomic<uint32_t> configured[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint32_t bit = !split ? 1u : (clustered ? (deep ? 16u : 8u) : 2u);
    const uint32_t nonportable_bit = deep ? 32u : 4u;
    if (dev < 0 || dev >= kMaxDevices || !(configured[dev].load() & bit)) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) configured[dev].fetch_or(bit);
    }
    void* args[] = {const_cast<AttendParams*>(&p), const_cast<CUtensorMap*>(&maps[0]),
                    const_cast<CUtensorMap*>(&maps[1])};
    if (clustered && p.cluster > 8 &&
        (dev < 0 || dev >= kMaxDevices || !(configured[dev].load() & nonportable_bit))) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) configured[dev].fetch_or(nonportable_bit);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // Cluster merge: the grid.x = cluster partitions of a group form one cluster.
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = clustered ? (unsigned)p.cluster : 1u;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = clustered ? 2 : 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// Clusters of c CTAs (2 .. kMaxClusterParts) of the cluster-merge instance
// that the current device holds at once, for the planner: the exact figure
// for this device (its SM count and GPC layout), where a table measured on one
// part would only be a guess on another.
template <int D, typename T, bool ROPE>
cudaError_t attend_mma_cluster_occupancy(int c, int* clusters, bool deep) {
    const void* fn = reinterpret_cast<const void*>(&attend_mma_kernel<D, T, true, true, ROPE>);
    int smem = MmaCfg<D, ROPE>::kSmemBytes;
    if constexpr (kHasDeep<D, ROPE>) {
        if (deep) {
            fn = reinterpret_cast<const void*>(&attend_mma_kernel<D, T, true, true, ROPE, true>);
            smem = MmaCfg<D, ROPE, true>::kSmemBytes;
        }
    } else if (deep) {
        return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (c > 8) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)c, 1, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(clusters, fn, &cfg);
}

// Launchers of the plain instances and of the rotary ones (fp16 / bf16 each).
template <int D, typename T>
cudaError_t launch_attend_mma_d(bool split, const AttendParams& p, const CUtensorMap* maps,
                                dim3 grid, cudaStream_t stream) {
    return launch_attend_mma_dr<D, T, false>(split, p, maps, grid, stream);
}

template <int D, typename T>
cudaError_t launch_attend_mma_rope_d(bool split, const AttendParams& p, const CUtensorMap* maps,
                                     dim3 grid, cudaStream_t stream) {
    return launch_attend_mma_dr<D, T, true>(split, p, maps, grid, stream);
}

}  // namespace pa
