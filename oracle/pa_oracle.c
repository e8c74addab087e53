/*
 * pa_oracle.c -- fp64 CPU oracle for paged-KV grouped-query decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * bench's cpu_baseline / reference arm may load this.  The CUDA path shares no
 * code with it and never calls it.
 *
 * What it computes (the plain definition, no partitions, no online softmax):
 * one query token per sequence attends over that sequence's context, which is
 * stored in fixed-size pages reached through a block table.
 *
 *   for every sequence b and query head h:
 *     kvh   = h / g,  g = Hq / Hkv          (contiguous head groups; the
 *                                           [kv_h, gqa, ...] -> [H, ...] reshape
 *                                           in the paged_attention_v2_pytorch.py
 *                                           commit note, GQA broadcast section)
 *     L     = context_lens[b]
 *     start = (window > 0 && window < L) ? L - window : 0
 *                                          (sliding window: the last `window`
 *                                           positions; apache/tvm PR #20426,
 *                                           section Correctness)
 *     for t in [start, L):
 *        page = block_tables[b][t / page_size], slot = t % page_size
 *        K_t  = k_cache[page][kvh][slot][:],  V_t likewise
 *                                          (gather through the page table,
 *                                           key_cache[blk_ids] in the commit note)
 *        s_t  = scale * sum_d q[b][h][d] * K_t[d]
 *     M   = max_t s_t,  Z = sum_t exp(s_t - M),  lse = M + ln Z
 *     out = sum_t exp(s_t - lse) * V_t     (softmax-weighted sum of V; the
 *                                           per-partition statistics and the
 *                                           log-sum-exp merge of the commit
 *                                           note's Phase 1 / Phase 2 reach
 *                                           exactly this value)
 *   L == 0 (nothing attended): out = 0, lse = -inf.
 *
 * Rotary embedding inside the kernel (rotary_mode = 1 of apache/tvm PR #20426,
 * section Correctness), when rope_theta > 0: before the scores, q is rotated
 * to position L - 1 (the new token) and every gathered K_t to position t, with
 * the rotate-half pairing of dimension i and i + D/2 and frequency
 * theta_i = rope_theta^(-2i/D):
 *     x'_i       = x_i cos(pos theta_i) - x_{i+D/2} sin(pos theta_i)
 *     x'_{i+D/2} = x_{i+D/2} cos(pos theta_i) + x_i sin(pos theta_i)
 * V is not rotated.
 *
 * Arithmetic: every fp16, bf16 or fp32 value is converted exactly to double
 * (binary16, bfloat16 and binary32 all embed exactly in binary64), all sums and
 * exponentials are in double.  `scale` is taken as a double.  No blocking,
 * reordering or fusion beyond the definition.
 *
 * Parity status: pinned (dense textbook attention, closed forms, invariants;
 * see tests/test_oracle_pins.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define PA_ORACLE_OK 0
#define PA_ORACLE_BAD_ARG 1
#define PA_ORACLE_BAD_PAGE 2
#define PA_ORACLE_NO_MEM 3

/* IEEE 754 binary16 -> binary64, exact: value = (-1)^s * 2^(e-15) * (1 + m/1024)
 * for 0 < e < 31, (-1)^s * 2^-14 * (m/1024) for e == 0, inf/nan for e == 31. */
static double half_bits_to_double(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1f;
    const int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);              /* 2^-14 * m / 2^10 */
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + m), e - 25);  /* 2^(e-15) * (1024+m) / 2^10 */
    }
    return sign ? -v : v;
}

double pa_oracle_half_to_double(uint16_t h) { return half_bits_to_double(h); }

/* bfloat16 -> binary64, exact: a bfloat16 is the upper 16 bits of a binary32
 * (sign, 8-bit exponent, 7-bit fraction), so value = (-1)^s * 2^(e-127) *
 * (1 + m/128) for 0 < e < 255, (-1)^s * 2^-126 * (m/128) for e == 0. */
static double bf16_bits_to_double(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int e = (h >> 7) & 0xff;
    const int m = h & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -133);             /* 2^-126 * m / 2^7 */
    } else if (e == 255) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(128 + m), e - 134);  /* 2^(e-127) * (128+m) / 2^7 */
    }
    return sign ? -v : v;
}

double pa_oracle_bf16_to_double(uint16_t h) { return bf16_bits_to_double(h); }

/* Element e of an array of the given type, exactly as a double. */
static double elem(const void* base, size_t e, int dtype) {
    if (dtype == 2) return (double)((const float*)base)[e];
    const uint16_t bits = ((const uint16_t*)base)[e];
    return dtype == 1 ? bf16_bits_to_double(bits) : half_bits_to_double(bits);
}

/* Rotate x[0..D) in place to position pos (rotate-half pairing). */
static void rope_rotate(double* x, int D, double theta, double pos) {
    const int half = D / 2;
    for (int i = 0; i < half; ++i) {
        const double freq = pow(theta, -2.0 * i / D);
        const double c = cos(pos * freq), sn = sin(pos * freq);
        const double a = x[i], b = x[i + half];
        x[i] = a * c - b * sn;
        x[i + half] = b * c + a * sn;
    }
}

/*
 * q            [B, Hq, D]                    binary16, bfloat16 or binary32
 * k_cache      [num_pages, Hkv, page_size, D] same element type
 * v_cache      same as k_cache
 * block_tables [B, max_pages_per_seq]         int32 physical page ids
 * context_lens [B]                            int32
 * out          [B, Hq, D]  double (written)
 * lse          [B, Hq]     double (written)
 * num_threads  OpenMP threads over (b, h); <= 0 means the runtime default.
 * dtype        element type of q, k_cache, v_cache: 0 = fp16, 1 = bf16, 2 = fp32.
 * rope_theta   > 0: rotary embedding of q and K as above; 0: none.
 * Returns 0, or a PA_ORACLE_* code (a page id outside [0, num_pages) or a
 * context longer than the table are reported, never read).
 */
int pa_oracle_decode(int B, int Hq, int Hkv, int D, int page_size, int num_pages,
                     int max_pages_per_seq, const void* q, const void* k_cache,
                     const void* v_cache, const int32_t* block_tables,
                     const int32_t* context_lens, double scale, int window, double* out,
                     double* lse, int num_threads, int dtype, double rope_theta) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || page_size <= 0 ||
        num_pages < 0 || max_pages_per_seq < 0 || dtype < 0 || dtype > 2 ||
        (rope_theta > 0 && D % 2 != 0))
        return PA_ORACLE_BAD_ARG;
    const int g = Hq / Hkv;
    int status = PA_ORACLE_OK;

#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif

#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < (long)B * Hq; ++bh) {
        const int b = (int)(bh / Hq);
        const int h = (int)(bh % Hq);
        const int kvh = h / g;
        const int L = context_lens[b];
        double* o = out + ((size_t)b * Hq + h) * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (L < 0 || (long)L > (long)max_pages_per_seq * page_size) {
#pragma omp atomic write
            status = PA_ORACLE_BAD_ARG;
            lse[(size_t)b * Hq + h] = NAN;
            continue;
        }
        const int start = (window > 0 && window < L) ? L - window : 0;
        const int n = L - start;
        if (n == 0) {
            lse[(size_t)b * Hq + h] = -INFINITY;
            continue;
        }
        double* s = (double*)malloc(sizeof(double) * (size_t)n);
        double* qd = (double*)malloc(sizeof(double) * (size_t)D);
        double* kd = (double*)malloc(sizeof(double) * (size_t)D);
        if (!s || !qd || !kd) {
            free(s);
            free(qd);
            free(kd);
#pragma omp atomic write
            status = PA_ORACLE_NO_MEM;
            continue;
        }
        const size_t qrow = ((size_t)b * Hq + h) * D;
        for (int d = 0; d < D; ++d) qd[d] = elem(q, qrow + d, dtype);
        if (rope_theta > 0) rope_rotate(qd, D, rope_theta, (double)(L - 1));

        int bad = 0;
        /* Step 1-2: gather K_t through the table, score it. */
        for (int t = start; t < L && !bad; ++t) {
            const int page = block_tables[(size_t)b * max_pages_per_seq + t / page_size];
            if (page < 0 || page >= num_pages) {
                bad = 1;
                break;
            }
            const size_t krow = (((size_t)page * Hkv + kvh) * page_size + (t % page_size)) * D;
            for (int d = 0; d < D; ++d) kd[d] = elem(k_cache, krow + d, dtype);
            if (rope_theta > 0) rope_rotate(kd, D, rope_theta, (double)t);
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += qd[d] * kd[d];
            s[t - start] = scale * dot;
        }
        if (bad) {
            free(s);
            free(qd);
            free(kd);
#pragma omp atomic write
            status = PA_ORACLE_BAD_PAGE;
            lse[(size_t)b * Hq + h] = NAN;
            continue;
        }
        /* Step 3: max, exp-sum, log-sum-exp. */
        double M = -INFINITY;
        for (int i = 0; i < n; ++i)
            if (s[i] > M) M = s[i];
        double Z = 0.0;
        for (int i = 0; i < n; ++i) Z += exp(s[i] - M);
        const double l = M + log(Z);
        lse[(size_t)b * Hq + h] = l;
        /* Step 4: softmax-weighted sum of the gathered V rows. */
        for (int t = start; t < L; ++t) {
            const int page = block_tables[(size_t)b * max_pages_per_seq + t / page_size];
            const size_t vrow = (((size_t)page * Hkv + kvh) * page_size + (t % page_size)) * D;
            const double w = exp(s[t - start] - l);
            for (int d = 0; d < D; ++d) o[d] += w * elem(v_cache, vrow + d, dtype);
        }
        free(s);
        free(qd);
        free(kd);
    }
    return status;
}

/* Scores alone (scale * q . K_t for t in [start, L)) for one (b, h), in the same
 * arithmetic as pa_oracle_decode; used by tests that check the log-sum-exp
 * identity against an independent library routine.  Returns the number of
 * scores written to s_out (capacity cap), or -1 on a bad page / argument. */
int pa_oracle_scores(int Hq, int Hkv, int D, int page_size, int num_pages, int max_pages_per_seq,
                     const void* q, const void* k_cache, const int32_t* block_tables,
                     const int32_t* context_lens, double scale, int window, int b, int h,
                     double* s_out, int cap, int dtype, double rope_theta) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || dtype < 0 || dtype > 2 || D > 1024) return -1;
    const int kvh = h / (Hq / Hkv);
    const int L = context_lens[b];
    if (L < 0 || (long)L > (long)max_pages_per_seq * page_size) return -1;
    const int start = (window > 0 && window < L) ? L - window : 0;
    if (L - start > cap) return -1;
    const size_t qrow = ((size_t)b * Hq + h) * D;
    double qd[1024], kd[1024];
    for (int d = 0; d < D; ++d) qd[d] = elem(q, qrow + d, dtype);
    if (rope_theta > 0) rope_rotate(qd, D, rope_theta, (double)(L - 1));
    for (int t = start; t < L; ++t) {
        const int page = block_tables[(size_t)b * max_pages_per_seq + t / page_size];
        if (page < 0 || page >= num_pages) return -1;
        const size_t krow = (((size_t)page * Hkv + kvh) * page_size + (t % page_size)) * D;
        for (int d = 0; d < D; ++d) kd[d] = elem(k_cache, krow + d, dtype);
        if (rope_theta > 0) rope_rotate(kd, D, rope_theta, (double)t);
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qd[d] * kd[d];
        s_out[t - start] = scale * dot;
    }
    return L - start;
}
