/*
 * bsp.h — C ABI of the block-sparse paged attention library (libbsp.so).
 *
 * The operation (FlashInfer: Making Attention Fit the Serving Workload, §2.1
 * eq 1 and §3.1 eq 4-5): for every query row i of request b and query head h,
 *
 *     s_j  = sm_scale * <q[i, h], k_j>          over the allowed keys j
 *     LSE  = log sum_j exp(s_j)                 (natural log)
 *     O    = sum_j exp(s_j - LSE) v_j
 *
 * where k_j, v_j come from kv head floor(h / g), g = H_qo / H_kv (same page,
 * §2.2 eq 3), and the keys of request b are its logical tokens 0..kv_len-1
 * found through a block-sparse (BSR) page table (same page, §4.1 eq 7):
 *
 *     page = kv_indices[kv_indptr[b] + t / page_size]
 *     row  = page * page_size + t % page_size
 *     kv_len = (kv_indptr[b+1] - kv_indptr[b] - 1) * page_size + last_page_len[b]
 *
 * With causal = 1 the mask is bottom-right aligned: query i of a request with
 * qo_len rows sees key j iff j <= i + kv_len - qo_len (FlashInfer 原理
 * overview, ⑧). A row with no allowed key gets O = 0 and LSE = -inf.
 *
 * The call sequence is the pages' plan/run split (FlashInfer: A Customizable
 * Attention Engine for LLM Serving, §6 and §8; technical review §6.3-6.4):
 *
 *   1. Once: size and allocate a device workspace (bsp_workspace_size) and a
 *      pinned host staging buffer (bsp_host_staging_size) for fixed upper
 *      bounds (bsp_capacity).
 *   2. Per generation step, on the host: bsp_plan() turns the request lengths
 *      into a load-balanced work list and a reduction map, writes them to the
 *      staging buffer and queues one async copy into the workspace on `stream`.
 *   3. Per layer, on the device: bsp_decode_run() or bsp_prefill_run() runs the
 *      attention kernel over the plan and then the merge of split outputs. The
 *      launch shape and every pointer are fixed by the plan info and the
 *      workspace, so a run can be captured in a CUDA graph and replayed after
 *      later plans into the same workspace.
 *   4. bsp_merge_state() merges two sets of attention states (shared-prefix
 *      composition).
 *
 * Conventions, common to every entry point:
 *   - Return value: BSP_OK (0) or a negative BSP_ERR_*; bsp_last_error()
 *     then gives a message (thread-local). Nothing is thrown across the ABI.
 *   - Every pointer is owned by the caller. Device pointers are plain CUDA
 *     device addresses of the current device; host pointers are plain host
 *     memory. No entry point allocates device memory; bsp_plan allocates only
 *     small host scratch. The run calls take q, k_pages, v_pages, o and the
 *     workspace 16-byte aligned (BSP_ERR_INVALID_ARG otherwise).
 *   - Layouts (row-major, innermost last):
 *       q, o          [n_tokens, H_qo, D]      ragged, no padding
 *       lse           [n_tokens, H_qo]         float32, natural log
 *       k_pages,
 *       v_pages       [num_pages, page_size, H_kv, D]   ("NHD" pages)
 *     dtype of q, k, v and o: BSP_DTYPE_BF16 or BSP_DTYPE_F32 (all the same).
 *   - All device work is queued on `stream` in stream order. The workspace
 *     and staging buffers must outlive every run (and graph replay) that uses
 *     them; the staging buffer must not be overwritten while the copy of the
 *     previous plan is still pending on its stream.
 */
#ifndef BSP_H_
#define BSP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *bsp_stream_t; /* same type as cudaStream_t */

/* ---- status codes ---------------------------------------------------- */
#define BSP_OK                  0
#define BSP_ERR_INVALID_ARG   (-1) /* malformed metadata or arguments          */
#define BSP_ERR_CAPACITY      (-2) /* plan exceeds the workspace's bounds      */
#define BSP_ERR_CUDA          (-3) /* a CUDA call failed                       */
#define BSP_ERR_UNSUPPORTED   (-4) /* shape or dtype the kernels do not cover  */
#define BSP_ERR_DEVICE_CHECK  (-5) /* a kernel's bounded wait or check tripped */

/* ---- enums ----------------------------------------------------------- */
#define BSP_DTYPE_BF16 0
#define BSP_DTYPE_F32  1

/* Work schedules of the plan (bsp_capacity.schedule). */
#define BSP_SCHEDULE_LPT          0 /* the pages' plan: chunks of L tokens, longest first onto the least-loaded CTA */
#define BSP_SCHEDULE_EQUAL_SHARES 1 /* not on the pages: equal contiguous shares of the concatenated KV ranges */

#define BSP_MODE_DECODE  0 /* query tile = the g fused heads of one position */
#define BSP_MODE_PREFILL 1 /* query tile = 256 packed rows (two MMA subtiles) */

/* Static problem description: what stays fixed across steps and layers. */
typedef struct bsp_problem {
    int32_t mode;          /* BSP_MODE_DECODE or BSP_MODE_PREFILL                 */
    int32_t num_qo_heads;  /* H_qo                                                 */
    int32_t num_kv_heads;  /* H_kv; H_qo % H_kv == 0, g = H_qo / H_kv             */
    int32_t head_dim;      /* D: 64 or 128 (prefill: 128)                         */
    int32_t page_size;     /* B_c >= 1                                            */
    int32_t causal;        /* 0 or 1, bottom-right aligned                        */
    int32_t dtype;         /* BSP_DTYPE_BF16 or BSP_DTYPE_F32 (prefill: BF16)      */
    /* Variants (FlashInfer 原理 overview, ⑧; FlashInfer: Making Attention Fit the
     * Serving Workload, eq 8). Zero-initialised problems get neither.           */
    int32_t window_left;   /* sliding window: query i sees key j only if
                              j >= i + kv_len - qo_len - window_left; 0 or
                              negative: no window (as -1)                         */
    float logits_soft_cap; /* c > 0: scores s become c * tanh(s / c) (s already
                              scaled by sm_scale) before masking and softmax;
                              0: none                                            */
    /* Attention sink (FlashInfer 原理 overview, ⑧, the AttentionSink variant):
     * device, float [H_qo], one logit per query head that joins every row's
     * softmax normaliser without a value row:
     *     LSE = log(exp(sink[h]) + sum_j exp(s_j)),  O = sum_j exp(s_j - LSE) v_j
     * (a row with no visible key: O = 0, LSE = sink[h]). NULL: none. Read at
     * run time from the plan's copy of the problem, so a plan shared by layers
     * may point it at each layer's sinks between runs. Not owned.              */
    const float *sink;
} bsp_problem;

/* Upper bounds fixed when the workspace is sized (technical review §6.4:
 * persistent buffers sized to declared bounds; exceeding them is an error). */
typedef struct bsp_capacity {
    int32_t max_batch;      /* requests per plan                                  */
    int32_t num_ctas;       /* plan queues C: the LPT plan balances C queues. The
                               kernels launch min(C, R) CTAs for R resident CTAs
                               of the device when C is a multiple of R or at most
                               R; otherwise each CTA runs ceil(C / R) consecutive
                               queues, so C = R + 1 .. 2R - 1 leaves SMs idle:
                               prefer R (bsp_default_num_ctas) or a multiple  */
    int64_t max_qo_tokens;  /* total query positions per plan                     */
    int32_t chunks_per_cta; /* s >= 1 (0 reads as 1): the chunk length becomes
                               L = ceil(W / (s C)), about s chunks per queue, so
                               that LPT can even out batches of few, equal tiles
                               (s = 1 is the pages' L = ceil(W / C)). Bounds the
                               work items by tiles + s C and the partial slots
                               by 2 s C; at most 64                            */
    int32_t max_gather_pages; /* prefill only (0 in decode): pages of the K / V
                               copy region the workspace reserves, each pool
                               max_gather_pages x page_size x H_kv x D
                               elements. 0: no region. With a region, a prefill
                               run whose pages the TMA page gather cannot take
                               (pages under 8 tokens or not a power of two)
                               and whose page table has at most this many
                               pages (kv_indptr[batch]) first copies the
                               table's pages, in table order, into the region
                               and then reads every request's keys as one
                               contiguous run of rows by TMA. That costs one
                               read and one write of the table's K and V, and
                               pays when each KV token is read by several
                               query tiles (long prefills); larger tables run
                               the cp.async gather as without a region      */
    int32_t schedule;       /* BSP_SCHEDULE_LPT (0, the pages' plan) or
                               BSP_SCHEDULE_EQUAL_SHARES (1; not on the pages):
                               the output tiles' visible KV ranges are laid end
                               to end in (request, tile, kv head) order and CTA
                               c takes the share [floor(c V / C),
                               floor((c + 1) V / C)) of the V tokens, a cut
                               inside a tile moved down to a page boundary. A
                               tile's pieces between cuts are its chunks (its
                               partial slots in order, as for LPT); an empty
                               tile's one chunk goes to the first CTA whose share
                               ends after its position. Every CTA gets the same
                               KV (to within a page) in at most a few items:
                               for batches of few, equal tiles, where LPT over
                               whole tiles leaves CTAs idle. chunks_per_cta is
                               ignored; the bounds hold with s = 1           */
} bsp_capacity;

/* One work item of the plan (64 bytes, device and staging image). */
typedef struct bsp_work_item {
    int32_t b;            /* request                                            */
    int32_t tile;         /* query tile within the request                      */
    int32_t kv_head;      /* kv head                                            */
    int32_t kv_start;     /* first logical KV token of the chunk                */
    int32_t kv_end;       /* one past the last logical KV token of the chunk    */
    int32_t slot;         /* partial-state slot, or -1: write the final output  */
    int32_t q_tok0;       /* global index of the tile's first query position    */
    int32_t n_pos;        /* query positions in the tile                        */
    int32_t qo_len;       /* query positions of request b                       */
    int32_t kv_len;       /* KV tokens of request b                             */
    int32_t page_base;    /* kv_indptr[b]                                       */
    int32_t pos0;         /* tile's first query position within the request     */
    int32_t merge;        /* reduction-map entry of `slot`, or -1                */
    int32_t reserved[3];
} bsp_work_item;

/* One entry of the reduction map (32 bytes): an output tile whose state is
 * the left-to-right merge of partial slots slot_begin .. slot_begin+n_slots-1. */
typedef struct bsp_merge_entry {
    int32_t b, tile, kv_head;
    int32_t slot_begin, n_slots;
    int32_t q_tok0, n_pos;
    int32_t arrived;      /* device-side count of this entry's partial states
                             written in the current run (0 when the plan is
                             copied, and again after a run's merge)             */
} bsp_merge_entry;

/* Host-side description of a plan (filled by bsp_plan, passed to the runs). */
typedef struct bsp_plan_info {
    bsp_problem problem;
    bsp_capacity capacity;
    int32_t batch;
    int32_t tile_rows;      /* T_q packed rows per query tile                     */
    int32_t group;          /* g                                                  */
    int32_t chunk_len;      /* L: maximum KV tokens per chunk (equal shares: the
                               longest chunk of the plan)                         */
    int64_t total_work;     /* W                                                  */
    int64_t alpha, beta;    /* cost = alpha * positions + beta * chunk tokens     */
    int32_t num_items;
    int32_t num_merges;     /* entries of the reduction map                       */
    int32_t num_partials;
    int32_t cap_items, cap_merges, cap_partials;
    /* byte offsets of the sections inside the workspace (and, for the metadata
     * sections, inside the staging buffer, which has the same layout up to
     * off_partial_lse) */
    uint64_t off_header, off_queue_indptr, off_items, off_merges;
    uint64_t off_status;     /* device error word (not part of the copied plan) */
    uint64_t off_partial_lse, off_partial_o;
    uint64_t metadata_bytes; /* bytes copied host -> device per plan          */
    uint64_t workspace_bytes;
    int32_t valid;           /* 1: planned and copied; 2: host-only plan      */
    int32_t num_qo_tokens;   /* qo_indptr[batch]: rows of q and o             */
    int32_t num_table_pages; /* kv_indptr[batch]: entries of kv_indices used  */
    int32_t reserved0;
    uint64_t off_gather;     /* K copy region (the V region follows it at
                                off_gather + gather_pool_bytes), 0 if none   */
    uint64_t gather_pool_bytes;
} bsp_plan_info;

/* Number of persistent CTAs the attention kernel of `mode` wants on `device`
 * (SM count x resident CTAs per SM). */
int bsp_default_num_ctas(int32_t mode, int32_t device, int32_t *num_ctas_out);

/* Bytes of device workspace for these bounds: plan metadata plus partial
 * states. Partial slots are bounded by 2 s C (technical review §6.5 eq 13, per
 * query tile and kv head). Returns 0 on invalid input. */
size_t bsp_workspace_size(const bsp_problem *problem, const bsp_capacity *capacity);

/* Bytes of the (pinned) host staging buffer for these bounds. */
size_t bsp_host_staging_size(const bsp_problem *problem, const bsp_capacity *capacity);

/*
 * Plan one step (FlashInfer 原理 overview, ⑨; technical review §6.1-6.2
 * Algorithm 2; engineering walkthrough §VIII.2, §VIII.5):
 *   query tiles of T_q packed rows (decode: g rows, one position; prefill:
 *   256 rows), W = sum over (tile, kv head) of kv_len, chunk length
 *   L = ceil(W / (s C)) rounded up to a page (s = capacity->chunks_per_cta), chunks of each tile's visible range
 *   sorted longest first (ties by (b, tile, kv_head, kv_start)), assigned to
 *   CTAs by a min-heap on (cost, cta), cost += alpha * positions + beta *
 *   chunk tokens; outputs with one chunk are written through, the others get
 *   consecutive partial slots merged left to right.
 *
 *   batch            number of requests B (<= capacity->max_batch)
 *   qo_indptr_h      host, int32 [B+1]; NULL in decode mode means one query
 *                    per request (qo_indptr = 0, 1, ..., B)
 *   kv_indptr_h      host, int32 [B+1], pages of each request
 *   last_page_len_h  host, int32 [B], 1..page_size for requests with pages
 *   alpha, beta      cost coefficients (the pages' default: 2 and 1)
 *   host_staging     host buffer of bsp_host_staging_size() bytes (pinned, so
 *                    that the copy is asynchronous)
 *   workspace        device buffer of bsp_workspace_size() bytes, or NULL to
 *                    plan on the host only (the plan is then only in
 *                    host_staging and nothing is queued; such a plan cannot run)
 *   stream           the copy staging -> workspace is queued on it
 *   out              filled on success
 * Errors: BSP_ERR_INVALID_ARG for malformed metadata (indptr not monotone,
 * last_page_len out of range, lengths beyond int32), BSP_ERR_CAPACITY when the
 * plan needs more items, merges, partial slots, requests or query positions
 * than the bounds allow (nothing is written then), BSP_ERR_CUDA if the copy
 * cannot be queued.
 */
int bsp_plan(const bsp_problem *problem, const bsp_capacity *capacity, int32_t batch,
             const int32_t *qo_indptr_h, const int32_t *kv_indptr_h,
             const int32_t *last_page_len_h, int64_t alpha, int64_t beta,
             void *host_staging, void *workspace, size_t workspace_bytes,
             bsp_stream_t stream, bsp_plan_info *out);

/*
 * Decode run: split-KV attention with the g heads of a kv head fused into one
 * tile (engineering walkthrough §II.4; overview ⑦). Split outputs are merged
 * over the reduction map (walkthrough §VIII.4-5) inside the same kernel: each
 * CTA that writes a partial state counts it in the output's reduction-map
 * entry, and the CTA whose partial completes the count folds them all (no CTA
 * waits for another). One launch.
 *   plan        from bsp_plan with mode BSP_MODE_DECODE
 *   q           device, [n_tokens, H_qo, D]
 *   k_pages,
 *   v_pages     device, [num_pages, page_size, H_kv, D]
 *   kv_indices  device, int32, the page ids (same array the plan's indptr
 *               indexes); may be NULL when no request has a page
 *   num_pages   pages in the k_pages / v_pages pools: bounds the tensor maps
 *               of the TMA page gather (pages of 8 or more tokens); 0 when
 *               unknown, which gathers with cp.async instead; < 0 is
 *               BSP_ERR_INVALID_ARG
 *   sm_scale    score scale (usually 1/sqrt(D))
 *   o           device, [n_tokens, H_qo, D], written
 *   lse         device, float [n_tokens, H_qo], written; may be NULL
 *   workspace   the workspace the plan was copied into
 * Supported: bf16 with D in {64, 128} and g <= 16; fp32 with D <= 256.
 */
int bsp_decode_run(const bsp_plan_info *plan, const void *q, const void *k_pages,
                   const void *v_pages, const int32_t *kv_indices, int64_t num_pages,
                   float sm_scale, void *o, float *lse, void *workspace, bsp_stream_t stream);

/*
 * Decode run over an e4m3 (FP8) KV cache (the e4m3 KV-cache configuration of
 * FlashInfer: A Customizable Attention Engine for LLM Serving, App. G.4
 * Table 8). Keys and values are stored as OCP e4m3 bytes with one scale per
 * pool: k = k_scale * k8, v = v_scale * v8. Everything else is bsp_decode_run
 * with those k and v; queries and outputs stay bf16, scores and the state are
 * fp32, and the converted values are exact (every e4m3 value is a bf16 value).
 *   plan        from bsp_plan with mode BSP_MODE_DECODE and dtype bf16
 *   q           device, bf16 [n_tokens, H_qo, 128]
 *   k_pages,
 *   v_pages     device, e4m3 bytes [num_pages, page_size, H_kv, 128]
 *   num_pages   pages in each pool, > 0 (bounds the tensor maps)
 *   k_scale,
 *   v_scale     finite, > 0
 *   o, lse, kv_indices, workspace: as for bsp_decode_run
 * Supported: head_dim 128, g <= 16, page_size a power of two >= 8. Anything
 * else is BSP_ERR_UNSUPPORTED (shape) or BSP_ERR_INVALID_ARG (scales, pool).
 */
int bsp_decode_run_fp8(const bsp_plan_info *plan, const void *q, const void *k_pages,
                       const void *v_pages, const int32_t *kv_indices, int64_t num_pages,
                       float sm_scale, float k_scale, float v_scale, void *o, float *lse,
                       void *workspace, bsp_stream_t stream);

/*
 * Prefill run: ragged queries, tiles of 256 packed rows (positions x g heads,
 * technical review eq 3) against KV tiles gathered page by page into shared
 * memory, QK^T and PV on the tensor cores (sparse gather, dense compute:
 * overview ⑥, walkthrough §IV.2 and §V.4), then the merge of split outputs.
 *   num_pages   pages in the k_pages / v_pages pools (bounds of the gather)
 *   other arguments as in bsp_decode_run.
 * Supported: bf16, D = 128, 128 % g == 0; pages of 8 or more tokens (powers of
 * two) are gathered with TMA tensor copies, other page sizes with cp.async.
 */
int bsp_prefill_run(const bsp_plan_info *plan, const void *q, const void *k_pages,
                    const void *v_pages, const int32_t *kv_indices, int64_t num_pages,
                    float sm_scale, void *o, float *lse, void *workspace, bsp_stream_t stream);

/*
 * The two stages of a run, for callers that time or schedule them apart
 * (bsp_prefill_run is exactly these two calls in order; bsp_decode_run is the
 * first alone, and the second after it recomputes the same merged outputs):
 *   bsp_run_attention       the attention kernel over the plan's work items
 *                           (final outputs for unsplit tiles, partial states in
 *                           the workspace for split ones, which decode also
 *                           merges in the same kernel); num_pages as in
 *                           bsp_decode_run / bsp_prefill_run
 *   bsp_run_merge_partials  the merge of partial states over the reduction map
 *                           (engineering walkthrough §VIII.4, the contraction
 *                           kernel); it always launches, with a fixed grid, and
 *                           does nothing when the plan split no output.
 */
int bsp_run_attention(const bsp_plan_info *plan, const void *q, const void *k_pages,
                      const void *v_pages, const int32_t *kv_indices, int64_t num_pages,
                      float sm_scale, void *o, float *lse, void *workspace, bsp_stream_t stream);
int bsp_run_merge_partials(const bsp_plan_info *plan, void *o, float *lse, void *workspace,
                           bsp_stream_t stream);

/*
 * Merge two sets of attention states (technical review §3.2 eq 6 and §3.3
 * Algorithm 1): with m = max(LSE_a, LSE_b), a = e^(LSE_a - m), b = e^(LSE_b - m),
 *   O = (a O_a + b O_b) / (a + b),   LSE = m + log(a + b);
 * a state with LSE = -inf is empty: it passes the other through; two empty
 * states give O = 0, LSE = -inf.
 *   o_a, o_b, o_out    device, [n_rows, num_heads, head_dim] in `dtype`
 *   lse_a, lse_b,
 *   lse_out            device, float [n_rows, num_heads]
 * o_out / lse_out may alias o_a / lse_a (in-place). head_dim <= 256.
 */
int bsp_merge_state(const void *o_a, const float *lse_a, const void *o_b, const float *lse_b,
                    void *o_out, float *lse_out, int64_t n_rows, int32_t num_heads,
                    int32_t head_dim, int32_t dtype, bsp_stream_t stream);

/*
 * Decode run without any device allocation by the caller or the library.
 *
 * The paper has no counterpart: this is a convenience of this library. It is
 * for callers that cannot call cudaMalloc where they run attention: a serving
 * engine whose KV-cache manager reserved nearly all of HBM for its own pool
 * and forbids further allocation while serving, or a plugin that its host
 * hands only input and output tensors, with no allocator for scratch. The
 * caller plans as usual (bsp_plan, where `workspace` may be NULL for a
 * host-only plan) and passes the plan and its staging image; this call copies
 * the plan into a fixed device array owned by the library, uses that array
 * as the workspace (plan metadata and partial states), runs the decode kernel
 * with its merge of split outputs, and allocates nothing.
 *
 *   plan          from bsp_plan, mode BSP_MODE_DECODE; its workspace_bytes
 *                 must not exceed BSP_STATIC_WORKSPACE_BYTES (else
 *                 BSP_ERR_CAPACITY: lower capacity.num_ctas or max_batch);
 *                 counts and offsets that do not match the layout of its
 *                 problem and capacity are BSP_ERR_INVALID_ARG
 *   host_staging  the staging buffer that bsp_plan wrote this plan into; the
 *                 copies out of it are queued on `stream`, so it must stay
 *                 unchanged until they have run (pinned memory makes them
 *                 asynchronous; pageable memory is copied before return)
 *   other arguments as in bsp_decode_run (device pointers, caller-owned);
 *   the pool size is not passed, so pages are gathered with cp.async, and
 *   the result is bit for bit that of bsp_decode_run with num_pages = 0 on
 *   the same plan.
 *
 * The array (BSP_STATIC_WORKSPACE_BYTES of device memory) exists once per
 * device in every process that loads the library and lives until the
 * process exits. The first call on a device looks its address up
 * (cudaGetSymbolAddress), so make that first call before any stream capture.
 * All calls on a device share the one array and it keeps the previous
 * call's contents: calls whose work may overlap on the GPU (two streams, or
 * two host threads) race on it and must be serialised by the caller, e.g.
 * by using one stream.
 */
#define BSP_STATIC_WORKSPACE_BYTES (8u << 20)
int bsp_decode_run_static(const bsp_plan_info *plan, const void *host_staging, const void *q,
                          const void *k_pages, const void *v_pages, const int32_t *kv_indices,
                          float sm_scale, void *o, float *lse, bsp_stream_t stream);

/* Self-test of the bounded waits every kernel uses: one warp waits on an
 * mbarrier that nothing arrives at, with the kernels' spin (polls, and every
 * 256 polls a clock and abort-flag check) and a limit of limit_cycles SM clock
 * cycles (1 .. 2^33, about 4 s); when it gives up it writes 0x1ff into *status (device
 * int32, set to 0 by the caller first) with the same compare-and-swap the
 * kernels use on the workspace status word, and the kernel returns: no fault,
 * the context stays usable. Stream-ordered; BSP_OK once launched. */
int bsp_check_bounded_wait(int64_t limit_cycles, int32_t *status, bsp_stream_t stream);

/* Read (and clear) the device error word that kernels set when a bounded wait
 * gives up or a bounds check trips (it lives in the workspace section at
 * plan->off_status). Synchronises `stream`. *word_out = 0 when clean;
 * otherwise it holds the code of the first check that tripped, and the
 * arrival counts of the plan's reduction map (bsp_merge_entry.arrived, which
 * CTAs that gave up may have left part-way) are reset to 0 as well, so the
 * same plan in the same workspace can run again. Outputs of the failed run
 * are undefined. */
int bsp_check_device_error(const bsp_plan_info *plan, void *workspace, bsp_stream_t stream,
                           int32_t *word_out);

/* Message for the last error on this thread ("" if none). */
const char *bsp_last_error(void);

/* Library version string. */
const char *bsp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BSP_H_ */
