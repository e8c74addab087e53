/*
 * pa.h -- C ABI of the GB300 paged-KV grouped-query decode-attention library
 * (libpa_gb300.so, built for sm_103a).
 *
 * One query token per sequence attends over that sequence's context, stored in
 * fixed-size pages of a KV cache reached through a block (page) table, with
 * grouped-query heads: Hq = g * Hkv and query head h reads KV head h / g (the
 * [kv_h, gqa, ...] -> [H, ...] grouping of the paged_attention_v2_pytorch.py
 * commit note, GQA broadcast section).  The attended context of each sequence
 * is cut into partitions; each partition yields a partial output and its
 * (max, exp-sum), and a log-sum-exp merge combines the partitions into the
 * final output and LSE (the commit note's Phase 1 and Phase 2).  When one
 * partition covers the whole attended context the kernel writes the output
 * directly and no merge runs (the short-context nest kept by apache/tvm PR
 * #20426, section Change).
 *
 * Result computed, for sequence b and query head h (natural log):
 *   start = (window > 0 && window < L_b) ? L_b - window : 0
 *   s_t   = scale * q[b,h,:] . K_t   for t in [start, L_b)
 *   lse   = log sum_t exp(s_t);   out = sum_t exp(s_t - lse) * V_t
 * L_b == 0 (or an empty attended range) gives out = 0, lse = -inf.
 *
 * Layouts (row-major, element strides implied by the shapes):
 *   q            T     [B, Hq, D]      T = fp16, bf16 or fp32 (plan.dtype)
 *   k_cache      T     [num_pages, Hkv, page_size, D]   (v_cache the same)
 *   block_tables int32 [B, max_pages_per_seq]   entry j = physical page of the
 *                                               sequence's logical page j
 *   context_lens int32 [B]
 *   out          T     [B, Hq, D]   (round to nearest even)
 *   lse          fp32  [B, Hq]
 * Supported: head_dim in {64, 96, 128, 256} (96 with the tensor-core kernel
 * only, fp32 with the CUDA-core kernel only); page_size 16;
 * Hq % Hkv == 0 with g = Hq / Hkv split into at most ceil(g / 8) equal head
 * chunks per CTA.
 * q, k_cache, v_cache, out and workspace must be 16-byte aligned.
 *
 * Ownership: every pointer is caller-owned device memory.  No call allocates
 * or frees device memory.  Two things are held by the library itself: the
 * fixed scratch array behind pa_decode_static (a __device__ array of
 * PA_STATIC_WORKSPACE_BYTES on every GPU that loads the library), and small
 * per-thread host caches (tensor-map encodings of the last K/V pools, the
 * last rotary frequency table).  Calls are asynchronous on the given stream
 * (a cudaStream_t passed as void*; NULL = the legacy default stream) and
 * never synchronise the host, except pa_get_error and pa_get_error_ex.
 *
 * Errors: every call returns a pa_status.  Argument checks happen on the host
 * before anything is launched.  Data-dependent faults found on the device (a
 * page id outside [0, num_pages), a context length outside
 * [0, max_context_len] or longer than the table) are never read through: the
 * kernel sets a bit in the workspace's device error word (pa_get_error) and
 * writes NaN to the affected output rows.
 */
#ifndef PA_GB300_H
#define PA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad shape or inconsistent plan */
    PA_ERR_UNSUPPORTED = 2,   /* valid but not built: head_dim, page_size, group size */
    PA_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    PA_ERR_WORKSPACE = 4      /* workspace missing or smaller than plan.workspace_bytes */
} pa_status;

/* Bits of the device error word (pa_get_error). */
#define PA_DEVERR_BAD_PAGE 1u     /* a block-table entry outside [0, num_pages) */
#define PA_DEVERR_BAD_LENGTH 2u   /* a context length outside the plan's bounds */
#define PA_DEVERR_TIMEOUT 4u      /* a bounded wait on a bulk copy gave up */

typedef struct pa_plan {
    int batch;              /* B */
    int num_q_heads;        /* Hq */
    int num_kv_heads;       /* Hkv */
    int head_dim;           /* D */
    int page_size;          /* tokens per page (16) */
    int num_pages;          /* pages in the K (and V) pool */
    int max_pages_per_seq;  /* row length of block_tables */
    int max_context_len;    /* upper bound on every context_lens[b] */
    int window;             /* sliding window in tokens, 0 = whole context */
    int partition_size;     /* tokens per partition, a multiple of page_size */
    int num_partitions;     /* partitions per (sequence, KV head); 1 = no split, no merge */
    int heads_per_cta;      /* query heads one CTA serves (g or a divisor of it) */
    int num_sms;            /* SM count the plan was made for */
    int ctas;               /* CTAs of the attention kernel (INT_MAX if more);
                               informational */
    size_t workspace_bytes; /* bytes of device workspace pa_decode needs (enough for
                               one partial per partition, whatever parts_per_cta) */
    int kernel;             /* PA_KERNEL_* used for the partition kernel; pa_plan picks
                               one, a caller may overwrite it before pa_decode */
    int parts_per_cta;      /* consecutive partitions one CTA of the tensor-core kernel
                               serves, 1, 2 or 4 (each gets 4 / parts_per_cta warps);
                               the CTA merges them (log-sum-exp) into one partial, so
                               each head has ceil(num_partitions / parts_per_cta)
                               partials.  The CUDA-core kernel always serves one */
    int merge_in_kernel;    /* 1: with the tensor-core kernel, the last CTA of each
                               (sequence, KV head) merges that group's partials and
                               pa_merge has nothing to do; 0: pa_merge launches the
                               merge kernel.  pa_plan_ex sets 1 for fixed partitions of
                               up to 8 partials per group, for rotary plans whose
                               group partials fit 128 KiB, and for work-balanced plans
                               as described under balanced */
    int ctrl_bytes;         /* leading workspace bytes that must be zero before the
                               first call (error word, per-group arrival counters).
                               Every call leaves the counters zero; the error word
                               keeps its bits until pa_get_error_ex clears them.  A
                               plan edited after pa_plan is rejected when this no
                               longer covers its counters */
    int dtype;              /* PA_DTYPE_*: element type of q, k_cache, v_cache and out
                               (pa_plan sets fp16; a caller may set bf16 or fp32) */
    float rope_theta;       /* > 0: rotary embedding inside the kernel (rotate-half
                               pairing of dim i and i + D/2, frequency
                               rope_theta^(-2i/D); q at position L - 1, K_t at t, V
                               untouched): the tensor-core kernel (fp16, bf16) or the
                               CUDA-core kernel (fp16, bf16, fp32); 0 = none */
    int cluster;            /* > 1: with the tensor-core kernel, the num_partitions
                               (== cluster, at most 16) CTAs of each (sequence, KV head,
                               head chunk) run as one thread-block cluster and merge the
                               group's partials through distributed shared memory, so
                               pa_decode_partitions writes out and lse itself and
                               pa_merge has nothing to do (parts_per_cta must be 1 and
                               merge_in_kernel 0); 0 or 1: no cluster */
    int prewait_prefetch;   /* tensor-core kernel: pages per warp (0 = off, at most 8)
                               requested into L2 before the wait for the grid this call
                               depends on (programmatic dependent launch).  Each CTA reads
                               its sequence length and first page ids as hints for them;
                               everything is read again after the wait, so a stale hint
                               only prefetches a page that is not used.  pa_plan_ex sets 2,
                               which pays when the preceding kernel on the stream is a
                               decode step (or any kernel that launches dependents
                               early): the hints then run while it drains.  Behind a
                               kernel that does not, 0 is faster (the hints' two
                               dependent reads come before this call's own) */
    int test_stall_bytes;   /* test hook, 0 in normal use.  > 0 (at most 4096): in the
                               tensor-core kernel each warp's first page copy expects
                               this many bytes more than it carries, so the bounded
                               wait on it runs out (after 1 s): the call then takes its
                               copy-timeout path (PA_DEVERR_TIMEOUT, NaN rows) without
                               any fault.  Lets a test exercise that path */
    int balanced;           /* > 0: work-balanced partitions (tensor-core kernel).  The
                               grid has `balanced` CTAs (X) per (KV head, head chunk),
                               shared by the whole batch, and the partition size is
                               chosen on the device from the actual context lengths:
                               with T the batch's attended pages, every partition has
                               pp = clamp(ceil(T / (X - B)), 8, 256) pages and sequence
                               b gets max(1, ceil(pages_b / pp)) CTAs, so a long
                               sequence gets more CTAs than a short one.  Its partials
                               are merged by the last CTA of each group
                               (merge_in_kernel = 1) or by the merge kernel (0);
                               pa_plan_ex takes the merge kernel when one group could
                               leave its last CTA more than 128 KiB of partials to
                               merge.  cluster 0, parts_per_cta 1.
                               num_partitions then holds X (the most partials a
                               sequence can have) and partition_size the largest pp
                               any lengths within max_context_len can give.  Set by
                               pa_plan_ex: with partition_size PA_PARTITION_BALANCED,
                               or automatically for a batch of several sequences
                               whose automatic plan would be a fixed split (not a
                               cluster merge, not unsplit); 0 = fixed-size
                               partitions */
    int deep_ring;          /* 1: with a cluster (tensor-core kernel, no rotary
                               embedding, head_dim 96, 128 or 256), the instance with
                               deeper page rings at 2 CTAs per SM instead of 3 (at
                               head_dim 256: 1 instead of 2), for cluster grids that do
                               not fill the GPU: a CTA streaming alone on its SM is
                               bound by what its own ring keeps in flight.  pa_plan_ex
                               sets it when the grid has at most one CTA per SM (at
                               head_dim 256 at most one per two SMs) and one wave of the
                               instance holds every cluster; 0 otherwise.  Ignored without a cluster; with one, 1 is
                               rejected for other kernels, head dims or rotary plans */
} pa_plan_t;

/* pa_plan / pa_plan_ex partition_size: work-balanced partitions sized on the
 * device (pa_plan_t.balanced); PA_ERR_UNSUPPORTED where none can be made. */
#define PA_PARTITION_BALANCED (-1)

/* Element types (pa_plan_t.dtype).  fp16 and bf16 run on either kernel, fp32
 * on the CUDA-core kernel only (fp32 FMA throughout; head_dim 64/128/256). */
#define PA_DTYPE_F16 0
#define PA_DTYPE_BF16 1
#define PA_DTYPE_F32 2

/* Partition-kernel variants (pa_plan_t.kernel). */
#define PA_KERNEL_SIMT 1   /* fp32 FMA on CUDA cores; pages by 1-D bulk copies */
#define PA_KERNEL_MMA 2    /* mma.sync tensor cores (fp16/bf16 in, fp32 accumulate);
                              pages by TMA tensor copies with the 128-byte swizzle */

/*
 * Choose the partitioning for a decode call (host only, no device access
 * unless num_sms == 0, which queries the current device).
 *   partition_size  0 = automatic (enough partitions to fill num_sms SMs),
 *                   PA_PARTITION_BALANCED = work-balanced partitions over the
 *                   batch (pa_plan_t.balanced), else the tokens per partition
 *                   (multiple of page_size).
 * The attended span of a sequence is at most ceil(max_context_len / ps) pages,
 * or ceil((window - 1) / ps) + 1 pages with a window; num_partitions =
 * ceil(span / (partition_size / ps)).  The 100000-token, 512-token-partition
 * case of the commit note therefore gets 196 partitions (the last one holds
 * 160 tokens).
 * Returns PA_OK and fills *plan, or PA_ERR_INVALID_ARG / PA_ERR_UNSUPPORTED.
 */
int pa_plan(int batch, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
            int num_pages, int max_pages_per_seq, int max_context_len, int window,
            int partition_size, int num_sms, pa_plan_t* plan);

/*
 * pa_plan for a given element type, kernel and rotary base: the automatic
 * partitioning then sizes the grid for that kernel's residency.
 *   dtype       PA_DTYPE_F16 / PA_DTYPE_BF16 / PA_DTYPE_F32
 *   kernel      0 = automatic (the tensor-core kernel, or the CUDA-core kernel
 *               for fp32 or a rotary embedding), else PA_KERNEL_*
 *   rope_theta  0 = no rotary embedding, else its frequency base
 * pa_plan(...) is pa_plan_ex(..., PA_DTYPE_F16, 0, 0, plan).  Returns
 * PA_ERR_UNSUPPORTED for combinations no kernel is built for.
 */
int pa_plan_ex(int batch, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
               int num_pages, int max_pages_per_seq, int max_context_len, int window,
               int partition_size, int num_sms, int dtype, int kernel, float rope_theta,
               pa_plan_t* plan);

/*
 * Full decode step: the partition kernel (gather pages, q.K, per-partition
 * softmax statistics, P.V) and, when plan->num_partitions > 1, the
 * log-sum-exp merge.  `window` must equal plan->window.
 * workspace: >= plan->workspace_bytes of device memory whose first
 * plan->ctrl_bytes are zero before the first call (zero-fill it once when
 * allocated).  They hold the device error word and per-group arrival
 * counters; every call leaves the counters zero again, and the error word
 * keeps its bits until read with pa_get_error_ex(clear = 1).  The rest holds
 * the partition partials between the kernels (and, for a work-balanced plan,
 * the partition size its partition kernel chose).  A workspace reused with a
 * different plan must have the new plan's ctrl_bytes zeroed first (the
 * counters may then lie where the old plan kept partials).  Concurrent calls
 * must not share a workspace.
 */
int pa_decode(const pa_plan_t* plan, const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, const int32_t* context_lens, float scale, int window,
              void* out, float* lse, void* workspace, void* stream);

/*
 * The two halves of pa_decode, for callers (and the benchmark) that time or
 * schedule them separately.  pa_decode_partitions writes the partials to the
 * workspace, one per CTA along the partitions (its parts_per_cta partitions
 * already merged), or, with one partition, out and lse directly; pa_merge
 * reads them and writes out and lse (a no-op with one partition, or when the
 * partition kernel merged them itself: merge_in_kernel or a cluster).
 * Same arguments and rules as pa_decode.
 */
int pa_decode_partitions(const pa_plan_t* plan, const void* q, const void* k_cache,
                         const void* v_cache, const int32_t* block_tables,
                         const int32_t* context_lens, float scale, int window, void* out,
                         float* lse, void* workspace, void* stream);
int pa_merge(const pa_plan_t* plan, const int32_t* context_lens, void* out, float* lse,
             void* workspace, void* stream);

/*
 * pa_decode for callers that cannot allocate device memory when they decode:
 * an engine or plugin that is handed only its own input and output buffers and
 * has no allocator to draw on, or a latency-critical loop that must never enter
 * the allocator (cudaMalloc can synchronise the whole device).  The pages have
 * no counterpart: this is a convenience of the library, not a step of the
 * method.
 *
 * Same arguments, layouts and result as pa_decode, minus the workspace: the
 * partition partials go to a scratch array of PA_STATIC_WORKSPACE_BYTES
 * compiled into the library (a __device__ array, so every GPU that loads the
 * library keeps that much memory until the process exits).  Nothing is
 * allocated or freed by this call.
 *   - The plan is checked on the host first, by pa_decode's rules.  Then the
 *     workspace extent its launches use is worked out from its shapes (not
 *     read from its ctrl_bytes field); a plan whose workspace_bytes, extent
 *     or ctrl_bytes exceeds PA_STATIC_WORKSPACE_BYTES is rejected with
 *     PA_ERR_WORKSPACE.  A rejected call touches no device memory.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture on that device.
 *   - Every call first clears the control bytes this plan uses (error word
 *     and arrival counters) on `stream` with cudaMemsetAsync, since the
 *     previous call may have used another plan, then runs pa_decode on it.
 *   - All calls on a device share the one array, which keeps the previous
 *     call's contents: calls whose kernels overlap on the GPU (different
 *     streams, no ordering between them) race on it and must not be issued.
 *   - Data-dependent faults still produce NaN rows in out/lse; the device
 *     error word lives in the shared array and is not reported by this call.
 */
#define PA_STATIC_WORKSPACE_BYTES (32u << 20)
int pa_decode_static(const pa_plan_t* plan, const void* q, const void* k_cache,
                     const void* v_cache, const int32_t* block_tables,
                     const int32_t* context_lens, float scale, int window, void* out,
                     float* lse, void* stream);

/*
 * Synchronise `stream` and read the device error word kept in `workspace`
 * (PA_DEVERR_* bits, 0 = none) into *device_error.  The word is left as it
 * is: its bits accumulate over calls until pa_get_error_ex clears them.
 * Returns PA_ERR_INVALID_ARG for a null pointer, PA_ERR_CUDA if the copy or
 * the synchronisation fails.
 */
int pa_get_error(void* workspace, void* stream, int* device_error);

/*
 * pa_get_error with a choice to clear: the word is read into *device_error
 * and, when `clear` is non-zero, reset to 0 on `stream` (then synchronised),
 * so that the next read reports only faults of later calls.
 */
int pa_get_error_ex(void* workspace, void* stream, int clear, unsigned* device_error);

/* Static text for a pa_status value. */
const char* pa_status_string(int status);

/* Library version, (major << 16) | minor. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_GB300_H */
