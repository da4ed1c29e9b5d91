/*
 * FP64 CPU oracle for paged extend attention (chunked prefill) and KV append.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may build, load or call this code.  It shares
 * nothing with the CUDA library: no headers, no helpers, no tables.
 *
 * What it computes is the plain definition, written out with loops:
 *
 *  - Slot of logical key j of sequence b (page-table addressing; AstrAI
 *    "scalar paged prefill fallback and decode causal fix", paged KV cache,
 *    PagePool.bind_tasks and the page-table form of the decode kernel):
 *        slot(b, j) = kv_indices[kv_indptr[b] + j / page_size] * page_size
 *                     + j % page_size
 *
 *  - KV append, continuing inside the last partly filled page (AReno PR #642,
 *    "What does this PR do?", third bullet; AstrAI CudaBackend.fwd_prefill,
 *    the write k_buffer[layer, out_cache_loc] = k):
 *        out_cache_loc[t] = slot(b, P_b + t - qo_indptr[b])
 *        k_pool[out_cache_loc[t]] = k[t],  v_pool[...] = v[t]
 *
 *  - Extend attention over cached prefix plus own chunk with bottom-right
 *    causal alignment (AReno PR #642, "What does this PR do?": later chunks
 *    attend to the cached prefix as well as the current chunk; AstrAI CPU
 *    reference of paged prefill, where the causal offset is the KV length
 *    minus the query length).  For query row i of sequence b (position
 *    p = P_b + i) and query head h (KV head g = h / (Hq / Hkv)):
 *        visible keys  V = { j : lo <= j <= p },  lo = max(0, p - W + 1) if
 *                      a window W > 0 is given (W keys including the query's
 *                      own position), else 0
 *        s_j   = sm_scale * sum_d q[i,h,d] * K[slot(b,j), g, d]
 *        M     = max_{j in V} s_j,   Z = sum_{j in V} exp(s_j - M)
 *        out   = sum_{j in V} exp(s_j - M) / Z * V[slot(b,j), g, :]
 *        lse   = M + ln Z                         (natural log, scaled scores)
 *    A two-pass softmax (scores first, then the maximum, then the weights) is
 *    used on purpose: it is the definition, not the streaming form.
 *
 *  - Non-causal attention and explicit boolean masks (AstrAI
 *    attn_paged_prefill: `is_causal`, and `mask` of shape [batch, 1, q_len,
 *    kv_len] or [batch, kv_len], True = keep, indexed by the request-local
 *    query row and the request-local key; the prefill-with-mask regression
 *    test runs a 4-D causal-pattern mask with causality off).  The visible
 *    set becomes
 *        V = { j < L_b :  (causal ? j <= p and the window rule : true)
 *                         and (mask ? mask[b, h, i, j] : true) }
 *    with i = t - qo_indptr[b] the row inside the chunk.  A mask is given by
 *    its base and element strides for b, h and i (0 for a broadcast
 *    dimension; the key stride is 1) and its extents in i and j: a row
 *    i >= q extent (when the i stride is not 0) or a key j >= kv extent reads
 *    as False.  A window needs causal attention.
 *    sm_scale <= 0 selects 1/sqrt(head_dim) (AstrAI attn_paged_prefill
 *    parameter packing: a non-positive scale means the default).
 *    An empty visible set gives out = 0 and lse = -inf.
 *
 * bf16 inputs arrive as their 16-bit patterns and are widened exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    ORACLE_OK = 0,
    ORACLE_ERR_INVALID_ARG = 1,
    ORACLE_ERR_BAD_INDEX = 3,
    ORACLE_ERR_NOMEM = 7
};

static double widen_bf16(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Physical slot of logical key j of sequence b, or -1 if the page entry is
 * missing, negative or beyond the pool. */
static int64_t key_slot(const int32_t* kv_indptr, const int32_t* kv_indices, int b,
                        int64_t j, int page_size, int64_t num_pages)
{
    int64_t entry = j / page_size;
    int64_t n_entries = (int64_t)kv_indptr[b + 1] - (int64_t)kv_indptr[b];
    if (entry >= n_entries) return -1;
    int64_t page = kv_indices[(int64_t)kv_indptr[b] + entry];
    if (page < 0 || page >= num_pages) return -1;
    return page * page_size + j % page_size;
}

int oracle_version(void) { return 2; }

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* out_cache_loc for every new token of the batch. */
int oracle_out_cache_loc(int batch, const int32_t* qo_indptr, const int32_t* kv_indptr,
                         const int32_t* kv_indices, const int32_t* prefix_lens,
                         int page_size, int64_t num_pages, int64_t* out_cache_loc)
{
    if (batch < 0 || page_size < 1) return ORACLE_ERR_INVALID_ARG;
    for (int b = 0; b < batch; ++b) {
        int64_t P = prefix_lens[b];
        for (int64_t t = qo_indptr[b]; t < qo_indptr[b + 1]; ++t) {
            int64_t pos = P + (t - qo_indptr[b]);
            int64_t s = key_slot(kv_indptr, kv_indices, b, pos, page_size, num_pages);
            if (s < 0) return ORACLE_ERR_BAD_INDEX;
            out_cache_loc[t] = s;
        }
    }
    return ORACLE_OK;
}

/* pool[loc[t]] = src[t] for K and V; row = n_kv_heads * head_dim elements. */
int oracle_kv_append(int64_t n_tokens, int64_t row_elems, const uint16_t* k, const uint16_t* v,
                     const int64_t* out_cache_loc, uint16_t* k_pool, uint16_t* v_pool,
                     int64_t pool_slots)
{
    for (int64_t t = 0; t < n_tokens; ++t) {
        int64_t s = out_cache_loc[t];
        if (s < 0 || s >= pool_slots) return ORACLE_ERR_BAD_INDEX;
    }
    for (int64_t t = 0; t < n_tokens; ++t) {
        int64_t s = out_cache_loc[t];
        memcpy(k_pool + s * row_elems, k + t * row_elems, (size_t)row_elems * sizeof(uint16_t));
        memcpy(v_pool + s * row_elems, v + t * row_elems, (size_t)row_elems * sizeof(uint16_t));
    }
    return ORACLE_OK;
}

/* Is key j visible to query row i (position p) of sequence b, query head h? */
static int key_visible(int64_t j, int64_t L, int64_t p, int causal, int window,
                       const uint8_t* mask, int64_t mb, int64_t mh, int64_t mq, int64_t mq_len,
                       int64_t mkv_len, int b, int h, int64_t i)
{
    if (j < 0 || j >= L) return 0;
    if (causal) {
        if (j > p) return 0;
        if (window > 0 && j < p - window + 1) return 0;
    }
    if (mask) {
        if (j >= mkv_len) return 0;
        if (mq != 0 && i >= mq_len) return 0;
        if (!mask[b * mb + h * mh + i * mq + j]) return 0;
    }
    return 1;
}

/* Attention for a list of (token, head) rows with the general visibility
 * rule (causal or not, optional boolean mask).  sel_tok[r] is a row of q
 * (0 <= t < total_q), sel_head[r] a query head.  out is [n_sel, head_dim],
 * lse is [n_sel].  Returns ORACLE_ERR_BAD_INDEX if a needed page is missing. */
int oracle_attention_rows_masked(int batch, const int32_t* qo_indptr, const int32_t* kv_indptr,
                                 const int32_t* kv_indices, const int32_t* prefix_lens,
                                 const uint16_t* q, const uint16_t* k_pool,
                                 const uint16_t* v_pool, int64_t num_pages, int page_size,
                                 int n_q_heads, int n_kv_heads, int head_dim, int window,
                                 double sm_scale, int causal, const uint8_t* mask,
                                 int64_t mask_b_stride, int64_t mask_h_stride,
                                 int64_t mask_q_stride, int64_t mask_q_len, int64_t mask_kv_len,
                                 int64_t n_sel, const int64_t* sel_tok, const int32_t* sel_head,
                                 double* out, double* lse)
{
    if (batch < 0 || page_size < 1 || n_q_heads < 1 || n_kv_heads < 1 || head_dim < 1 ||
        n_q_heads % n_kv_heads != 0 || window < 0 || (!causal && window > 0) ||
        (mask && (mask_q_len < 0 || mask_kv_len < 0)))
        return ORACLE_ERR_INVALID_ARG;
    const int group = n_q_heads / n_kv_heads;
    const double scale = sm_scale > 0.0 ? sm_scale : 1.0 / sqrt((double)head_dim);
    const int64_t total_q = batch > 0 ? qo_indptr[batch] : 0;
    int status = ORACLE_OK;

#pragma omp parallel
    {
        double* scores = NULL;
        int64_t* keys = NULL;
        int64_t cap = 0;
        double* acc = (double*)malloc(sizeof(double) * (size_t)head_dim);
        double* qrow = (double*)malloc(sizeof(double) * (size_t)head_dim);
        if (!acc || !qrow) {
#pragma omp atomic write
            status = ORACLE_ERR_NOMEM;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_sel; ++r) {
            int st_now;
#pragma omp atomic read
            st_now = status;
            if (st_now != ORACLE_OK) continue;
            const int64_t t = sel_tok[r];
            const int h = sel_head[r];
            if (t < 0 || t >= total_q || h < 0 || h >= n_q_heads) {
#pragma omp atomic write
                status = ORACLE_ERR_INVALID_ARG;
                continue;
            }
            /* the sequence that owns row t */
            int b = 0;
            while (!(qo_indptr[b] <= t && t < qo_indptr[b + 1])) ++b;
            const int64_t i = t - qo_indptr[b];
            const int64_t p = (int64_t)prefix_lens[b] + i;
            const int64_t L = (int64_t)prefix_lens[b] + (qo_indptr[b + 1] - qo_indptr[b]);
            const int g = h / group;
            double* o = out + r * head_dim;
            if (L > cap) {
                free(scores);
                free(keys);
                cap = L;
                scores = (double*)malloc(sizeof(double) * (size_t)cap);
                keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)cap);
                if (!scores || !keys) {
#pragma omp atomic write
                    status = ORACLE_ERR_NOMEM;
                    cap = 0;
                    continue;
                }
            }
            /* the visible keys, in increasing order */
            int64_t n_vis = 0;
            for (int64_t j = 0; j < L; ++j)
                if (key_visible(j, L, p, causal, window, mask, mask_b_stride, mask_h_stride,
                                mask_q_stride, mask_q_len, mask_kv_len, b, h, i))
                    keys[n_vis++] = j;
            if (n_vis == 0) {
                for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
                lse[r] = -INFINITY;
                continue;
            }
            for (int d = 0; d < head_dim; ++d)
                qrow[d] = widen_bf16(q[(t * n_q_heads + h) * (int64_t)head_dim + d]);
            /* pass 1: scaled scores */
            int bad = 0;
            for (int64_t k = 0; k < n_vis; ++k) {
                int64_t s = key_slot(kv_indptr, kv_indices, b, keys[k], page_size, num_pages);
                if (s < 0) { bad = 1; break; }
                const uint16_t* krow = k_pool + (s * n_kv_heads + g) * (int64_t)head_dim;
                double dot = 0.0;
                for (int d = 0; d < head_dim; ++d) dot += qrow[d] * widen_bf16(krow[d]);
                scores[k] = scale * dot;
            }
            if (bad) {
#pragma omp atomic write
                status = ORACLE_ERR_BAD_INDEX;
                continue;
            }
            /* pass 2: maximum and normaliser */
            double M = -INFINITY;
            for (int64_t k = 0; k < n_vis; ++k) if (scores[k] > M) M = scores[k];
            double Z = 0.0;
            for (int64_t k = 0; k < n_vis; ++k) Z += exp(scores[k] - M);
            /* pass 3: weighted sum of values */
            for (int d = 0; d < head_dim; ++d) acc[d] = 0.0;
            for (int64_t k = 0; k < n_vis; ++k) {
                int64_t s = key_slot(kv_indptr, kv_indices, b, keys[k], page_size, num_pages);
                const uint16_t* vrow = v_pool + (s * n_kv_heads + g) * (int64_t)head_dim;
                double w = exp(scores[k] - M) / Z;
                for (int d = 0; d < head_dim; ++d) acc[d] += w * widen_bf16(vrow[d]);
            }
            for (int d = 0; d < head_dim; ++d) o[d] = acc[d];
            lse[r] = M + log(Z);
        }
        free(scores);
        free(keys);
        free(acc);
        free(qrow);
    }
    return status;
}

/* Bottom-right causal attention without a mask, for a list of rows. */
int oracle_attention_rows(int batch, const int32_t* qo_indptr, const int32_t* kv_indptr,
                          const int32_t* kv_indices, const int32_t* prefix_lens,
                          const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                          int64_t num_pages, int page_size, int n_q_heads, int n_kv_heads,
                          int head_dim, int window, double sm_scale,
                          int64_t n_sel, const int64_t* sel_tok, const int32_t* sel_head,
                          double* out, double* lse)
{
    return oracle_attention_rows_masked(batch, qo_indptr, kv_indptr, kv_indices, prefix_lens, q,
                                        k_pool, v_pool, num_pages, page_size, n_q_heads,
                                        n_kv_heads, head_dim, window, sm_scale, 1, NULL, 0, 0,
                                        0, 0, 0, n_sel, sel_tok, sel_head, out, lse);
}

/* Every row of the batch with the general visibility rule:
 * out [total_q, n_q_heads, head_dim], lse [total_q, n_q_heads]. */
int oracle_attention_masked(int batch, const int32_t* qo_indptr, const int32_t* kv_indptr,
                            const int32_t* kv_indices, const int32_t* prefix_lens,
                            const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                            int64_t num_pages, int page_size, int n_q_heads, int n_kv_heads,
                            int head_dim, int window, double sm_scale, int causal,
                            const uint8_t* mask, int64_t mask_b_stride, int64_t mask_h_stride,
                            int64_t mask_q_stride, int64_t mask_q_len, int64_t mask_kv_len,
                            double* out, double* lse)
{
    const int64_t total_q = batch > 0 ? qo_indptr[batch] : 0;
    const int64_t n = total_q * n_q_heads;
    int64_t* tok = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    int32_t* head = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    if (!tok || !head) { free(tok); free(head); return ORACLE_ERR_NOMEM; }
    for (int64_t t = 0; t < total_q; ++t)
        for (int h = 0; h < n_q_heads; ++h) {
            tok[t * n_q_heads + h] = t;
            head[t * n_q_heads + h] = h;
        }
    int st = oracle_attention_rows_masked(batch, qo_indptr, kv_indptr, kv_indices, prefix_lens,
                                          q, k_pool, v_pool, num_pages, page_size, n_q_heads,
                                          n_kv_heads, head_dim, window, sm_scale, causal, mask,
                                          mask_b_stride, mask_h_stride, mask_q_stride,
                                          mask_q_len, mask_kv_len, n, tok, head, out, lse);
    free(tok);
    free(head);
    return st;
}

/* Every row of the batch, bottom-right causal, no mask. */
int oracle_attention(int batch, const int32_t* qo_indptr, const int32_t* kv_indptr,
                     const int32_t* kv_indices, const int32_t* prefix_lens,
                     const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                     int64_t num_pages, int page_size, int n_q_heads, int n_kv_heads,
                     int head_dim, int window, double sm_scale, double* out, double* lse)
{
    return oracle_attention_masked(batch, qo_indptr, kv_indptr, kv_indices, prefix_lens, q,
                                   k_pool, v_pool, num_pages, page_size, n_q_heads, n_kv_heads,
                                   head_dim, window, sm_scale, 1, NULL, 0, 0, 0, 0, 0, out, lse);
}
