/*
 * Oracle: plain fp64 CPU attention over a paged (BSR) KV cache, and the exact
 * merge of attention states.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, calls or
 * includes this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg load it. It shares no code with the CUDA path.
 *
 * Every function is the definition written out, one output at a time, with no
 * blocking, fusion or reordering:
 *
 *   - attention (FlashInfer: Making Attention Fit the Serving Workload, §2.1
 *     eq 1): S = Q K^T * sm_scale + M, O = softmax(S) V, the mask M being 0 for
 *     allowed keys and -inf for forbidden ones;
 *   - attention state (same page, §3.1 eq 4-5): LSE = log sum_j exp(s_j), the
 *     natural log of the normaliser of the scaled scores, O normalised;
 *   - head-group mapping (same page, §2.2 eq 3): query head h reads kv head
 *     floor(h / g), g = H_qo / H_kv;
 *   - logical -> physical token (same page, §4.1 eq 7):
 *     p = indices[indptr[b] + floor(t / B_c)], row = p * B_c + (t mod B_c);
 *   - kv length of a request: (pages - 1) * B_c + last_page_len, 0 without
 *     pages (FlashInfer: A Customizable Attention Engine for LLM Serving, §8,
 *     the plan(page_indptr, page_indices, last_page_length, ...) call);
 *   - causal mask, bottom-right aligned: query i of a request with qo_len rows
 *     and kv_len keys sees key j iff j <= i + kv_len - qo_len (FlashInfer
 *     原理 overview, ⑧, the sink mask with the window term removed);
 *   - sliding window (FlashInfer 原理 overview, ⑧, the sink variant's mask):
 *     with window_left > 0, key j is also required to satisfy
 *     j + qo_len + window_left >= kv_len + i;
 *   - logits soft-cap (FlashInfer: Making Attention Fit the Serving Workload,
 *     eq 8): with c = soft_cap > 0 each allowed score becomes c * tanh(s / c),
 *     s being the scaled score, before the softmax;
 *   - attention sink (FlashInfer 原理 overview, ⑧, the AttentionSink variant:
 *     a per-head value enters the online softmax's (m, d) as one more logit
 *     and the output is normalised by that larger d): with sink != NULL,
 *     LSE = log(exp(sink[h]) + sum_j exp(s_j)) and O = sum_j exp(s_j - LSE) v_j;
 *     the sink has no value row, so a row with no visible key gets O = 0,
 *     LSE = sink[h];
 *   - stable merge with the empty-state rule (FlashInfer: Making Attention Fit
 *     the Serving Workload, §3.2 eq 6 and §3.3 Algorithm 1).
 *
 * Inputs are float (bf16 and fp32 values are exact in float); all arithmetic
 * is double. An empty key set gives O = 0, LSE = -inf (without a sink).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_INPUT (-1)

/* Length in tokens of request b's KV: full pages then the valid part of the
 * last page. */
static int64_t kv_len_of(const int32_t *kv_indptr, const int32_t *last_page_len,
                         int32_t page_size, int32_t b)
{
    int64_t npages = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
    if (npages <= 0) return 0;
    return (npages - 1) * page_size + last_page_len[b];
}

/* eq 7: physical token row of logical token t of request b. */
int64_t oracle_physical_row(const int32_t *kv_indptr, const int32_t *kv_indices,
                            int32_t page_size, int32_t b, int64_t t)
{
    int64_t page = kv_indices[kv_indptr[b] + t / page_size];
    return page * page_size + t % page_size;
}

/* Request that owns query token `tok` (qo_indptr is non-decreasing). */
static int32_t request_of_token(const int32_t *qo_indptr, int32_t batch, int64_t tok)
{
    int32_t lo = 0, hi = batch - 1;
    while (lo < hi) {
        int32_t mid = (lo + hi + 1) / 2;
        if (qo_indptr[mid] <= tok) lo = mid; else hi = mid - 1;
    }
    return lo;
}

/*
 * Attention for a list of (query token, query head) pairs.
 *
 *   q          [n_tokens, H_qo, D]           query rows (ragged, no padding)
 *   k_pages    [num_pages, page_size, H_kv, D]
 *   v_pages    [num_pages, page_size, H_kv, D]
 *   qo_indptr  [batch + 1]  query rows of request b: qo_indptr[b] .. qo_indptr[b+1]
 *   kv_indptr  [batch + 1]  pages of request b: kv_indices[kv_indptr[b] .. kv_indptr[b+1]]
 *   last_page_len [batch]   valid tokens in the last page, 1..page_size
 *   sel_token, sel_head [n_sel]  which outputs to compute
 *   o_out  [n_sel, D], lse_out [n_sel]   (double)
 */
int oracle_attention_rows(int32_t batch, int32_t H_qo, int32_t H_kv, int32_t D,
                          int32_t page_size, int32_t causal, double sm_scale,
                          int32_t window_left, double soft_cap, const double *sink,
                          const int32_t *qo_indptr, const int32_t *kv_indptr,
                          const int32_t *kv_indices, const int32_t *last_page_len,
                          const float *q, const float *k_pages, const float *v_pages,
                          int64_t n_sel, const int64_t *sel_token, const int32_t *sel_head,
                          double *o_out, double *lse_out, int32_t num_threads)
{
    if (batch < 1 || H_qo < 1 || H_kv < 1 || H_qo % H_kv != 0 || D < 1 || page_size < 1)
        return ORACLE_BAD_INPUT;
    const int32_t g = H_qo / H_kv;
#ifdef _OPENMP
    /* a thread count for this call only (omp_set_num_threads would outlive it) */
    const int n_threads = num_threads > 0 ? num_threads : omp_get_max_threads();
#else
    const int n_threads = 1;
    (void)num_threads;
#endif
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad) num_threads(n_threads)
    for (int64_t s = 0; s < n_sel; ++s) {
        const int64_t tok = sel_token[s];
        const int32_t h = sel_head[s];
        double *o = o_out + s * D;
        if (tok < 0 || tok >= qo_indptr[batch] || h < 0 || h >= H_qo) { bad = 1; continue; }
        const int32_t b = request_of_token(qo_indptr, batch, tok);
        const int64_t qo_len = (int64_t)qo_indptr[b + 1] - qo_indptr[b];
        const int64_t kv_len = kv_len_of(kv_indptr, last_page_len, page_size, b);
        const int64_t i = tok - qo_indptr[b];
        const int32_t hk = h / g;                                /* eq 3 */
        int64_t n_vis = kv_len;                                  /* keys j < n_vis are allowed */
        if (causal) {
            int64_t lim = i + kv_len - qo_len + 1;               /* j <= i + kv_len - qo_len */
            if (lim < n_vis) n_vis = lim;
            if (n_vis < 0) n_vis = 0;
        }
        int64_t j0 = 0;                                          /* keys j >= j0 are allowed */
        if (window_left > 0) {
            j0 = i + kv_len - qo_len - window_left;              /* j + qo_len + window_left >= kv_len + i */
            if (j0 < 0) j0 = 0;
        }
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
        if (n_vis <= j0) { lse_out[s] = sink ? sink[h] : -INFINITY; continue; }

        const float *qv = q + (tok * H_qo + h) * (int64_t)D;
        double *sc = (double *)malloc(sizeof(double) * (size_t)n_vis);
        if (!sc) { bad = 1; continue; }
        /* scores s_j = sm_scale * <q, k_j> (then capped: c * tanh(s_j / c)) */
        for (int64_t j = j0; j < n_vis; ++j) {
            int64_t row = oracle_physical_row(kv_indptr, kv_indices, page_size, b, j);
            const float *kv = k_pages + (row * H_kv + hk) * (int64_t)D;
            double acc = 0.0;
            for (int32_t d = 0; d < D; ++d) acc += (double)qv[d] * (double)kv[d];
            sc[j] = sm_scale * acc;
            if (soft_cap > 0.0) sc[j] = soft_cap * tanh(sc[j] / soft_cap);
        }
        /* LSE = m + log sum exp(s_j - m) */
        double m = sc[j0];
        for (int64_t j = j0 + 1; j < n_vis; ++j) if (sc[j] > m) m = sc[j];
        if (sink && sink[h] > m) m = sink[h];
        double z = 0.0;
        for (int64_t j = j0; j < n_vis; ++j) z += exp(sc[j] - m);
        if (sink) z += exp(sink[h] - m);                         /* the sink logit, no value row */
        const double lse = m + log(z);
        /* O = sum_j exp(s_j - LSE) v_j */
        for (int64_t j = j0; j < n_vis; ++j) {
            int64_t row = oracle_physical_row(kv_indptr, kv_indices, page_size, b, j);
            const float *vv = v_pages + (row * H_kv + hk) * (int64_t)D;
            const double p = exp(sc[j] - lse);
            for (int32_t d = 0; d < D; ++d) o[d] += p * (double)vv[d];
        }
        lse_out[s] = lse;
        free(sc);
    }
    return bad ? ORACLE_BAD_INPUT : ORACLE_OK;
}

/*
 * Stable merge of attention states, element-wise over n states of width D
 * (eq 6, Algorithm 1 of the technical review). A state with LSE = -inf is
 * empty: one empty side passes the other through; two empty sides stay empty
 * (O = 0, LSE = -inf).
 */
void oracle_merge_states(int64_t n, int32_t D,
                         const double *o_a, const double *lse_a,
                         const double *o_b, const double *lse_b,
                         double *o_out, double *lse_out)
{
    for (int64_t s = 0; s < n; ++s) {
        const double la = lse_a[s], lb = lse_b[s];
        const int va = !(isinf(la) && la < 0), vb = !(isinf(lb) && lb < 0);
        const double *oa = o_a + s * D, *ob = o_b + s * D;
        double *o = o_out + s * D;
        if (!va && !vb) {
            for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
            lse_out[s] = -INFINITY;
        } else if (!vb) {
            for (int32_t d = 0; d < D; ++d) o[d] = oa[d];
            lse_out[s] = la;
        } else if (!va) {
            for (int32_t d = 0; d < D; ++d) o[d] = ob[d];
            lse_out[s] = lb;
        } else {
            const double m = la > lb ? la : lb;
            const double a = exp(la - m), bb = exp(lb - m);
            for (int32_t d = 0; d < D; ++d) o[d] = (a * oa[d] + bb * ob[d]) / (a + bb);
            lse_out[s] = m + log(a + bb);
        }
    }
}

int oracle_num_threads_available(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
