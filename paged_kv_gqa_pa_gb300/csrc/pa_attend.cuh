// pa_attend.cuh -- the partition kernel of paged-KV GQA decode attention.
//
// One CTA serves one (partition, KV head, head chunk, sequence).  It walks the
// partition's pages of K and V through the block table (the page gather of the
// paged_attention_v2_pytorch.py commit note, key_cache[blk_ids]), loads each
// page once for all G query heads of its group (the commit note's GQA
// broadcast: K/V stay at kv-head size), and computes in fp32:
//   scores  s = scale * q.K        (Phase 1 QK^T)
//   softmax statistics (max, exp-sum) with an online update per page
//   P.V, the exp-weighted sum of the V rows
// It then writes either the partition's normalised output plus its (max,
// exp-sum) for the log-sum-exp merge (Phase 1 -> Phase 2 of the commit note;
// SPLIT = true), or, when one partition covers the whole attended context,
// the final fp16 output and the natural-log LSE (SPLIT = false; the
// short-context role of the tiled nest in apache/tvm PR #20426, section
// Change).
//
// GB300 mapping.  Four warps per CTA, each an independent pipeline: lane 0 of
// a warp streams that warp's pages (pages w, w+4, w+8, ... of the partition)
// with 1-D bulk copies (cp.async.bulk, one 16-token page of one KV head =
// 16*D*2 contiguous bytes) into a ring of kStages shared-memory slots guarded
// by mbarriers, so several pages per warp are in flight while the warp
// computes on an earlier one.  Within a warp a token row is covered by D/8
// lanes holding 16 bytes (8 dims) each; q for those 8 dims and G heads stays
// in registers, and the per-lane partial dot products are combined with a
// reduce-scatter of warp shuffles (each exchange halves the tokens a lane
// keeps), after which lane l holds the full scores of token l/2 of the page.
// The four warps' (max, exp-sum, output) states are merged in shared memory at
// the end, the same log-sum-exp algebra as the cross-partition merge.
#pragma once

#include <cuda_bf16.h>
#include <math.h>

#include <atomic>
#include <type_traits>

#include "pa_common.cuh"

namespace pa {

template <int D, int G>
struct Lanes {
    static constexpr int R = D / 8;   // lanes per token row, 8 dims each
    static constexpr int TL = R / 2;  // tokens of a page per lane
    static constexpr int LOG_TL = TL == 16 ? 4 : (TL == 8 ? 3 : (TL == 4 ? 2 : 0));
    static constexpr int GP = (G + 3) & ~3;  // row stride of the per-warp P buffer
    static_assert(D == 64 || D == 128 || D == 256, "head_dim");
    static_assert(R * kPageSize / 2 == D, "lane layout");
};

// Packed fp32 pair arithmetic: one fma.rn.f32x2 / mul.rn.f32x2 instruction
// (sm_100 and later) does the operation on both halves, which halves the
// issue slots of the lane-local rotations, dot products and P.V updates.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

// 8 packed 16-bit elements (fp16 or bf16) widened to 4 float pairs.
template <typename E>
__device__ __forceinline__ void wide8(const uint4 raw, float2 (&f)[4]);

template <>
__device__ __forceinline__ void wide8<__half>(const uint4 raw, float2 (&f)[4]) {
    const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
    for (int j = 0; j < 4; ++j) f[j] = __half22float2(h[j]);
}

template <>
__device__ __forceinline__ void wide8<__nv_bfloat16>(const uint4 raw, float2 (&f)[4]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int j = 0; j < 4; ++j) f[j] = __bfloat1622float2(h[j]);
}

// This lane's 8 consecutive elements starting at `src` (16 bytes of fp16 or
// bf16, 32 bytes of fp32), as 4 float pairs (dims 2j, 2j + 1 in f[j]).
template <typename E>
__device__ __forceinline__ void load8(const unsigned char* src, float2 (&f)[4]) {
    wide8<E>(*reinterpret_cast<const uint4*>(src), f);
}

template <>
__device__ __forceinline__ void load8<float>(const unsigned char* src, float2 (&f)[4]) {
    const float4 a = reinterpret_cast<const float4*>(src)[0];
    const float4 b = reinterpret_cast<const float4*>(src)[1];
    f[0] = make_float2(a.x, a.y);
    f[1] = make_float2(a.z, a.w);
    f[2] = make_float2(b.x, b.y);
    f[3] = make_float2(b.z, b.w);
}

template <typename E>
__device__ __forceinline__ E from_float_e(float v);
template <>
__device__ __forceinline__ __half from_float_e<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float_e<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Two floats packed into one 32-bit word of E (round to nearest even).
template <typename E>
__device__ __forceinline__ uint32_t pack2e(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2e<__half>(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2e<__nv_bfloat16>(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
template <>
__device__ __forceinline__ float from_float_e<float>(float v) { return v; }

// Four consecutive outputs of type E (8-byte aligned fp16/bf16, 16-byte fp32).
template <typename E>
__device__ __forceinline__ void store4e(E* dst, float a, float b, float c, float d) {
    if constexpr (sizeof(E) == 2) {
        uint2 packed;
        packed.x = pack2e<E>(a, b);
        packed.y = pack2e<E>(c, d);
        *reinterpret_cast<uint2*>(dst) = packed;
    } else {
        *reinterpret_cast<float4*>(dst) = make_float4(a, b, c, d);
    }
}


// Rotary state of a lane: cos and signed sin of its 8 frequencies at the
// position of the next token it scores, and the one-token step, as pairs
// (frequencies 2j, 2j + 1 in element j).  The lane's dims are [8r, 8r + 8) of
// the row; the lane r ^ (R/2) holds the partner dims (i <-> i + D/2 of the
// rotate-half pairing).  With sigma = -1 on the first half of the row and +1
// on the second, a rotated value is x cos + partner sigma sin, so every sine
// here carries sigma: the recurrence keeps its form because sigma^2 = 1.
struct RopeLane {
    float2 c[4], s[4];             // cos, sigma sin at the next position
    float2 c1[4], s1[4], ns1[4];   // one-token step: cos, sigma sin, -sigma sin
};

// (c, s) <- (c, s) turned by the angle whose (cos, sigma sin, -sigma sin) are
// (cr, sr, nsr): c' = c cr - s sr, s' = s cr + c sr.
__device__ __forceinline__ void rope_turn(float2& c, float2& s, float2 cr, float2 sr, float2 nsr) {
    const float2 cn = fma2(c, cr, mul2(s, nsr));
    const float2 sn = fma2(s, cr, mul2(c, sr));
    c = cn;
    s = sn;
}

// Rotate this lane's 8 K values (kf) with its partner's (pf) and advance the
// rotary state by one position.
__device__ __forceinline__ void rope_apply_and_step(float2 (&kf)[4], const float2 (&pf)[4],
                                                    RopeLane& rl) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        kf[j] = fma2(kf[j], rl.c[j], mul2(pf[j], rl.s[j]));
        rope_turn(rl.c[j], rl.s[j], rl.c1[j], rl.s1[j], rl.ns1[j]);
    }
}

// Partial dot products of the G heads with token `tok` of the K page (this
// lane's 8 dims), combined across the 2^LEVEL tokens tok .. tok + 2^LEVEL - 1
// by a shuffle reduce-scatter: the exchange over lane mask (1 << LEVEL) pairs
// token bit LEVEL-1, and a lane keeps the token whose bit equals its lane bit.
// Tokens are visited in increasing order, which the rotary recurrence relies on.
template <int D, int G, int LEVEL, typename E>
__device__ __forceinline__ void qk_tree(float (&res)[G], const unsigned char* kpage, int tok,
                                        int r, int lane, const float2 (&qf)[G][4], bool rope,
                                        RopeLane& rl) {
    if constexpr (LEVEL == 0) {
        const unsigned char* src = kpage + tok * (D * (int)sizeof(E)) + r * (8 * (int)sizeof(E));
        float2 kf[4];
        if (rope) {  // warp-uniform
            constexpr int kHalf = D / 16;  // lanes per half row
            float2 pf[4];
            if constexpr (sizeof(E) == 2) {
                // exchange the packed 16-bit words (4 shuffles), then widen
                const uint4 raw = *reinterpret_cast<const uint4*>(src);
                uint4 praw;
                praw.x = __shfl_xor_sync(0xffffffffu, raw.x, kHalf);
                praw.y = __shfl_xor_sync(0xffffffffu, raw.y, kHalf);
                praw.z = __shfl_xor_sync(0xffffffffu, raw.z, kHalf);
                praw.w = __shfl_xor_sync(0xffffffffu, raw.w, kHalf);
                wide8<E>(raw, kf);
                wide8<E>(praw, pf);
            } else {
                load8<E>(src, kf);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    pf[j].x = __shfl_xor_sync(0xffffffffu, kf[j].x, kHalf);
                    pf[j].y = __shfl_xor_sync(0xffffffffu, kf[j].y, kHalf);
                }
            }
            rope_apply_and_step(kf, pf, rl);
        } else {
            load8<E>(src, kf);
        }
        // even and odd dims accumulate in the two halves of a pair
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float2 a = mul2(qf[h][0], kf[0]);
#pragma unroll
            for (int j = 1; j < 4; ++j) a = fma2(qf[h][j], kf[j], a);
            res[h] = a.x + a.y;
        }
    } else {
        float lo[G], hi[G];
        qk_tree<D, G, LEVEL - 1, E>(lo, kpage, tok, r, lane, qf, rope, rl);
        qk_tree<D, G, LEVEL - 1, E>(hi, kpage, tok + (1 << (LEVEL - 1)), r, lane, qf, rope, rl);
        constexpr int kMask = 1 << LEVEL;
        const bool up = (lane & kMask) != 0;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float send = up ? lo[h] : hi[h];
            const float keep = up ? hi[h] : lo[h];
            res[h] = keep + __shfl_xor_sync(0xffffffffu, send, kMask);
        }
    }
}

template <int D, int G, bool SPLIT, typename E>
__device__ __forceinline__ void write_rows(const AttendParams& p, int b, int h0, int part,
                                           float o_val, float m_val, float l_val,
                                           float lse_val) {
    for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
        const int h = idx / D, d = idx % D;
        const size_t bh = (size_t)b * p.Hq + h0 + h;
        if constexpr (SPLIT) {
            const size_t row = bh * p.P + part;
            p.ws_o[row * D + d] = o_val;
            if (d == 0) {
                p.ws_m[row] = m_val;
                p.ws_l[row] = l_val;
            }
        } else {
            reinterpret_cast<E*>(p.out)[bh * D + d] = from_float_e<E>(o_val);
            if (d == 0) p.lse[bh] = lse_val;
        }
    }
}

template <int D, int G, bool SPLIT, bool ROPE, typename E>
__global__ void __launch_bounds__(kThreads, AttendCfg<D, sizeof(E)>::blocks_for(G))
    attend_kernel(const AttendParams p) {
    using Cfg = AttendCfg<D, sizeof(E)>;
    constexpr int ES = sizeof(E);
    using LN = Lanes<D, G>;
    constexpr int R = LN::R;
    constexpr int TL = LN::TL;
    constexpr int GP = LN::GP;
    constexpr int NS = Cfg::kStages;
    constexpr int PB = Cfg::kPageBytes;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem;                                         // [warps][NS][PB]
    float* pbuf = reinterpret_cast<float*>(smem + Cfg::kRingBytes);     // [warps][16][2 GP]
    int* s_pid = reinterpret_cast<int*>(pbuf + kWarps * Cfg::kPBufFloats);  // [kMaxPagesPerPart]
    float* s_ml = reinterpret_cast<float*>(s_pid + kMaxPagesPerPart);   // [warps][2][8]
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_ml + kWarps * kMaxHeadsPerCta * 2);
    __shared__ int s_flag;
    // rotary page turn per frequency: cos, sin, -sin
    __shared__ __align__(16) float s_rstep[ROPE ? 3 * (D / 2) : 4];
    static_assert(Cfg::blocks_for(G) * (Cfg::kSmemBytes + sizeof(s_rstep) + 16 + 1024) <=
                      228 * 1024,
                  "CTAs per SM by shared memory, static part included");

    // Programmatic dependent launch (see the tensor-core kernel).
    allow_dependent_launch();
    wait_for_prerequisite_grid();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int part = blockIdx.x;
    const int kvh = blockIdx.y / p.nchunk;
    const int h0 = kvh * p.g + (blockIdx.y % p.nchunk) * G;
    const int b = blockIdx.z;

    const SeqSpan sp = seq_span(p.context_lens[b], p.window, p.max_ctx, p.maxp, p.pages_per_part);
    if (!sp.valid) {
        if (threadIdx.x == 0 && part == 0 && blockIdx.y == 0) atomicOr(p.err, PA_DEVERR_BAD_LENGTH);
        if constexpr (!SPLIT) write_rows<D, G, SPLIT, E>(p, b, h0, part, NAN, NAN, NAN, NAN);
        return;  // with a split, the merge writes the NaN rows
    }
    if (part >= sp.num_parts) {
        // Nothing attended in this partition.  Without a split this only
        // happens for an empty context: out = 0, lse = -inf.
        if constexpr (!SPLIT) write_rows<D, G, SPLIT, E>(p, b, h0, part, 0.f, 0.f, 0.f, -INFINITY);
        return;
    }
    const int pg0 = sp.first_page + part * p.pages_per_part;
    const int npg = min(p.pages_per_part, sp.end_page - pg0);

    if (threadIdx.x == 0) s_flag = 0;
    const uint32_t bar_w = smem_u32(bars) + warp * NS * 8;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < NS; ++s) mbar_init(bar_w + s * 8, 1);
        fence_mbar_init();
    }
    __syncthreads();
    for (int j = threadIdx.x; j < npg; j += kThreads) {
        int id = p.block_tables[(size_t)b * p.maxp + pg0 + j];
        if (id < 0 || id >= p.num_pages) {
            s_flag = 1;
            id = 0;
        }
        s_pid[j] = id;
    }
    if constexpr (ROPE) {
        for (int i = threadIdx.x; i < D / 2; i += kThreads) {
            float c, sn;
            rope_twiddle(kWarps * kPageSize - TL, p.rope_phi[0][i], p.rope_phi[1][i], c, sn);
            s_rstep[i] = c;
            s_rstep[D / 2 + i] = sn;
            s_rstep[D + i] = -sn;
        }
    }
    __syncthreads();
    if (s_flag) {
        if (threadIdx.x == 0) atomicOr(p.err, PA_DEVERR_BAD_PAGE);
        write_rows<D, G, SPLIT, E>(p, b, h0, part, NAN, NAN, NAN, NAN);
        return;
    }

    // ---- this warp's pages: j = warp, warp + 4, ... ; items K0, V0, K1, V1, ...
    const int nk = npg > warp ? (npg - warp + kWarps - 1) / kWarps : 0;
    const int n_items = 2 * nk;
    const uint32_t ring_w = smem_u32(ring) + warp * NS * PB;
    const unsigned char* ring_wp = ring + warp * NS * PB;
    const size_t kv_stride = (size_t)kPageSize * D;  // elements per (page, kv head)

    auto issue = [&](int item) {
        const int slot = item % NS;
        const int jj = warp + (item >> 1) * kWarps;
        const unsigned char* base =
            reinterpret_cast<const unsigned char*>((item & 1) ? p.v : p.k);
        const unsigned char* src = base + ((size_t)s_pid[jj] * p.Hkv + kvh) * kv_stride * ES;
        const uint32_t bar = bar_w + slot * 8;
        mbar_arrive_expect_tx(bar, PB);
        bulk_g2s(ring_w + slot * PB, src, PB, bar);
    };
    int issued = 0;
    if (lane == 0) {
        for (int i = 0; i < NS && i < n_items; ++i) issue(i);
    }
    issued = min(NS, n_items);

    // ---- q for this lane's 8 dims, all G heads (fp32)
    const int r = lane % R;
    const int rg = lane / R;
    float2 qf[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        load8<E>(reinterpret_cast<const unsigned char*>(p.q) +
                     (((size_t)b * p.Hq + h0 + h) * D + r * 8) * ES,
                 qf[h]);
    }
    // Rotary embedding: q to position L - 1; the K rows follow per token.
    constexpr bool rope = ROPE;  // rotary instances are separate, so the plain ones pay nothing
    const float sigma = (r & (D / 16)) == 0 ? -1.f : 1.f;  // first / second half of the row
    const int rope_f0 = (r & (D / 16 - 1)) * 8;            // this lane's first frequency
    RopeLane rl;
    if (rope) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float c[2], sn[2], c1[2], s1[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int f = rope_f0 + 2 * j + e;
                rope_twiddle(1, p.rope_phi[0][f], p.rope_phi[1][f], c1[e], s1[e]);
                rope_twiddle(sp.L - 1, p.rope_phi[0][f], p.rope_phi[1][f], c[e], sn[e]);
            }
            rl.c1[j] = make_float2(c1[0], c1[1]);
            rl.s1[j] = make_float2(sigma * s1[0], sigma * s1[1]);
            rl.ns1[j] = make_float2(-sigma * s1[0], -sigma * s1[1]);
            rl.c[j] = make_float2(c[0], c[1]);
            rl.s[j] = make_float2(sigma * sn[0], sigma * sn[1]);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float2 pq[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                pq[j].x = __shfl_xor_sync(0xffffffffu, qf[h][j].x, D / 16);
                pq[j].y = __shfl_xor_sync(0xffffffffu, qf[h][j].y, D / 16);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) qf[h][j] = fma2(qf[h][j], rl.c[j], mul2(pq[j], rl.s[j]));
        }
    }
    // (cos, sigma sin, -sigma sin) of the turn from past this lane's tokens of
    // one page to its next page, from the shared table
    const float* rstep_s = s_rstep + (sigma < 0.f ? D : D / 2);
    const float* rstep_ns = s_rstep + (sigma < 0.f ? D / 2 : D);

    float2 o[G][4];
    float m[G], lsum[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        lsum[h] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) o[h][j] = make_float2(0.f, 0.f);
    }
    float* pw = pbuf + warp * Cfg::kPBufFloats;
    const int t_own = lane >> 1;  // token of the page whose scores this lane ends up with
    bool ok = true;
    int consumed = 0;

    for (int k = 0; k < nk; ++k) {
        // ---------------- K page: scores
        {
            const int item = 2 * k;
            const int slot = item % NS;
            const bool got = mbar_wait_bounded(bar_w + slot * 8, (item / NS) & 1);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            consumed = item + 1;
        }
        if (rope) {
            // Rotary state at this lane's first token of the page: evaluated
            // exactly every kRopeResync pages of this warp; in between, the
            // state the previous page's token recurrence left (TL tokens on)
            // is turned on to this page by one fixed rotation.
            constexpr int kRopeResync = 8;
            if (k % kRopeResync == 0) {
                const int pos0 = (pg0 + warp + k * kWarps) * kPageSize + rg * TL;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float c[2], sn[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int f = rope_f0 + 2 * j + e;
                        rope_twiddle(pos0, p.rope_phi[0][f], p.rope_phi[1][f], c[e], sn[e]);
                    }
                    rl.c[j] = make_float2(c[0], c[1]);
                    rl.s[j] = make_float2(sigma * sn[0], sigma * sn[1]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int f = rope_f0 + 2 * j;
                    rope_turn(rl.c[j], rl.s[j], *reinterpret_cast<const float2*>(s_rstep + f),
                              *reinterpret_cast<const float2*>(rstep_s + f),
                              *reinterpret_cast<const float2*>(rstep_ns + f));
                }
            }
        }
        float s[G];
        qk_tree<D, G, LN::LOG_TL, E>(s, ring_wp + ((2 * k) % NS) * PB, rg * TL, r, lane, qf, rope,
                                     rl);
#pragma unroll
        for (int h = 0; h < G; ++h) s[h] += __shfl_xor_sync(0xffffffffu, s[h], 1);
        __syncwarp();
        if (lane == 0 && 2 * k + NS < n_items) {
            fence_proxy_async_smem();
            issue(2 * k + NS);
        }
        if (2 * k + NS < n_items) issued = 2 * k + NS + 1;

        // ---------------- online softmax over this page (log2 domain)
        const int pos = (pg0 + warp + k * kWarps) * kPageSize + t_own;
        const bool valid = pos >= sp.start && pos < sp.L;
        float pm[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            s[h] = valid ? s[h] * p.scale_log2 : -INFINITY;
            pm[h] = s[h];
        }
#pragma unroll
        for (int mask = 2; mask < 32; mask <<= 1) {
#pragma unroll
            for (int h = 0; h < G; ++h) pm[h] = fmaxf(pm[h], __shfl_xor_sync(0xffffffffu, pm[h], mask));
        }
        bool grow = false;
#pragma unroll
        for (int h = 0; h < G; ++h) grow |= pm[h] > m[h];
        if (grow) {  // warp-uniform: every lane holds the same m and pm
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float mn = fmaxf(m[h], pm[h]);
                const float a = (mn == -INFINITY) ? 1.f : ex2(m[h] - mn);
                m[h] = mn;
                lsum[h] *= a;
#pragma unroll
                for (int j = 0; j < 4; ++j) o[h][j] = mul2(o[h][j], make_float2(a, a));
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float e = (s[h] == -INFINITY) ? 0.f : ex2(s[h] - m[h]);
            lsum[h] += e;
            s[h] = e;
        }
        // lanes 2t and 2t + 1 hold the same scores: each writes one half of
        // the (p, p) pairs the P.V step multiplies with
#pragma unroll
        for (int h = 0; h < G; ++h) pw[t_own * 2 * GP + 2 * h + (lane & 1)] = s[h];
        __syncwarp();

        // ---------------- V page: o += p * V
        {
            const int item = 2 * k + 1;
            const int slot = item % NS;
            const bool got = mbar_wait_bounded(bar_w + slot * 8, (item / NS) & 1);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            consumed = item + 1;
        }
        const unsigned char* vpage = ring_wp + ((2 * k + 1) % NS) * PB;
        const int vpos0 = (pg0 + warp + k * kWarps) * kPageSize;
        auto pv_page = [&](auto edge) {
#pragma unroll
            for (int i = 0; i < TL; ++i) {
                const int t = rg * TL + i;
                float2 vf[4];
                load8<E>(vpage + t * (D * ES) + r * (8 * ES), vf);
                // Slots outside [start, L) carry weight 0; zero their V too so
                // that whatever an unwritten slot holds (NaN included) cannot
                // leak in.  Only a page at an edge of the span has such slots.
                if constexpr (decltype(edge)::value) {
                    if (vpos0 + t < sp.start || vpos0 + t >= sp.L) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) vf[j] = make_float2(0.f, 0.f);
                    }
                }
                float2 pr[GP];
#pragma unroll
                for (int h2 = 0; h2 < GP; h2 += 2) {
                    const float4 t4 = *reinterpret_cast<const float4*>(pw + t * 2 * GP + 2 * h2);
                    pr[h2] = make_float2(t4.x, t4.y);
                    pr[h2 + 1] = make_float2(t4.z, t4.w);
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) o[h][j] = fma2(pr[h], vf[j], o[h][j]);
                }
            }
        };
        if (vpos0 < sp.start || vpos0 + kPageSize > sp.L)  // warp-uniform
            pv_page(std::true_type{});
        else
            pv_page(std::false_type{});
        __syncwarp();
        if (lane == 0 && 2 * k + 1 + NS < n_items) {
            fence_proxy_async_smem();
            issue(2 * k + 1 + NS);
        }
        if (2 * k + 1 + NS < n_items) issued = 2 * k + 1 + NS + 1;
    }

    if (!ok) {
        // A copy did not land in time: record it, give every copy this warp
        // issued a bounded chance to land (so none writes into shared memory
        // after the CTA exits), and publish NaN for this CTA.
        if (lane == 0) atomicOr(p.err, PA_DEVERR_TIMEOUT);
        for (int item = consumed; item < issued; ++item)
            (void)mbar_wait_bounded(bar_w + (item % NS) * 8, (item / NS) & 1);
        s_flag = 1;
    }

    // ---- combine lanes: exp-sums over the 16 tokens (lanes l and l^1 hold the
    // same token), outputs over the row groups of the warp.
#pragma unroll
    for (int mask = 2; mask < 32; mask <<= 1) {
#pragma unroll
        for (int h = 0; h < G; ++h) lsum[h] += __shfl_xor_sync(0xffffffffu, lsum[h], mask);
    }
#pragma unroll
    for (int mask = R; mask < 32; mask <<= 1) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                o[h][j].x += __shfl_xor_sync(0xffffffffu, o[h][j].x, mask);
                o[h][j].y += __shfl_xor_sync(0xffffffffu, o[h][j].y, mask);
            }
        }
    }
    __syncthreads();  // every warp is done with its ring: reuse it for the warp states
    float* s_o = reinterpret_cast<float*>(ring);  // [warps][G][D]
    if (lane < R) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float4* dst = reinterpret_cast<float4*>(s_o + (warp * G + h) * D + r * 8);
            dst[0] = make_float4(o[h][0].x, o[h][0].y, o[h][1].x, o[h][1].y);
            dst[1] = make_float4(o[h][2].x, o[h][2].y, o[h][3].x, o[h][3].y);
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            s_ml[warp * 2 * kMaxHeadsPerCta + h] = m[h];
            s_ml[warp * 2 * kMaxHeadsPerCta + kMaxHeadsPerCta + h] = lsum[h];
        }
    }
    __syncthreads();
    if (s_flag) {
        write_rows<D, G, SPLIT, E>(p, b, h0, part, NAN, NAN, NAN, NAN);
        return;
    }

    // ---- merge the four warp states (same log-sum-exp algebra as Phase 2)
    constexpr int D4 = D / 4;
    for (int idx = threadIdx.x; idx < G * D4; idx += kThreads) {
        const int h = idx / D4;
        const int d = (idx % D4) * 4;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_ml[w * 2 * kMaxHeadsPerCta + h]);
        float Ls = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float mw = s_ml[w * 2 * kMaxHeadsPerCta + h];
            const float c = (mw == -INFINITY) ? 0.f : ex2(mw - M);
            Ls += c * s_ml[w * 2 * kMaxHeadsPerCta + kMaxHeadsPerCta + h];
            const float4 ow = *reinterpret_cast<const float4*>(s_o + (w * G + h) * D + d);
            acc.x += c * ow.x;
            acc.y += c * ow.y;
            acc.z += c * ow.z;
            acc.w += c * ow.w;
        }
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        const size_t bh = (size_t)b * p.Hq + h0 + h;
        if constexpr (SPLIT) {
            const size_t row = bh * p.P + part;
            *reinterpret_cast<float4*>(p.ws_o + row * D + d) =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            if (d == 0) {
                p.ws_m[row] = M;
                p.ws_l[row] = Ls;
            }
        } else {
            store4e<E>(reinterpret_cast<E*>(p.out) + bh * D + d, acc.x * inv, acc.y * inv,
                       acc.z * inv, acc.w * inv);
            if (d == 0) p.lse[bh] = Ls > 0.f ? M * 0.69314718055994531f + logf(Ls) : -INFINITY;
        }
    }
}

// Launcher for one head dim and element type: picks the <G, SPLIT, ROPE>
// instance, raises its dynamic shared-memory limit once per device, launches
// on `stream`.
template <int D, typename E>
cudaError_t launch_attend_d(int G, bool split, const AttendParams& p, dim3 grid,
                            cudaStream_t stream) {
    using Cfg = AttendCfg<D, sizeof(E)>;
    const void* fn = nullptr;
    const bool rope = p.rope != 0;
    switch (G) {
#define PA_ATTEND_PICK(GG, S, R) reinterpret_cast<const void*>(&attend_kernel<D, GG, S, R, E>)
#define PA_ATTEND_CASE(GG)                                                                   \
    case GG:                                                                                 \
        fn = split ? (rope ? PA_ATTEND_PICK(GG, true, true) : PA_ATTEND_PICK(GG, true, false)) \
                   : (rope ? PA_ATTEND_PICK(GG, false, true) : PA_ATTEND_PICK(GG, false, false)); \
        break;
        PA_ATTEND_CASE(1)
        PA_ATTEND_CASE(2)
        PA_ATTEND_CASE(3)
        PA_ATTEND_CASE(4)
        PA_ATTEND_CASE(5)
        PA_ATTEND_CASE(6)
        PA_ATTEND_CASE(7)
        PA_ATTEND_CASE(8)
#undef PA_ATTEND_CASE
#undef PA_ATTEND_PICK
        default:
            return cudaErrorInvalidValue;
    }
    constexpr int kMaxDevices = 64;
    static std::atomic<uint32_t> configured[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint32_t bit = 1u << ((G - 1) * 4 + (split ? 2 : 0) + (rope ? 1 : 0));
    if (dev < 0 || dev >= kMaxDevices || !(configured[dev].load() & bit)) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) configured[dev].fetch_or(bit);
    }
    void* args[] = {const_cast<AttendParams*>(&p)};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace pa
