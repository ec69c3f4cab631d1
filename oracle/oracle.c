/*
 * oracle.c -- plain, slow, fp64 CPU oracle for attention over a paged KV pool.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark load this file's library.  The product path (the CUDA
 * library under paged_kv_cache_row_gb300/) never calls it and shares no code,
 * header, table or helper with it.
 *
 * What it computes, and where the pages define it:
 *   - store_kv: each new token's K and V row is copied into the pool at the
 *     physical row out_loc[i] ("mini-sglang-learn", paged KV pool section,
 *     store_kv passage: one token row scattered per new token, by out_loc).
 *   - attention of one query over a request's context, gathered through its
 *     page_table row, which holds raw physical row numbers
 *     ("mini-sglang architecture deep dive", section 3.6 TableManager page-table figure and
 *     section 5.3 PagedAttention figure; "mini-sglang-learn", page_table
 *     alignment passage).  The value is the textbook
 *         o = sum_j softmax_j(sm_scale * <q, K_j>) V_j
 *     with the max subtracted before exponentiation (section 5.2,
 *     FlashAttention: the same softmax, computed without tiling here).
 *   - decode: one query token per request, over logical tokens [0, seq_len).
 *   - extend: request r's new token t sits at absolute position
 *     cached_len[r] + t and sees logical tokens 0 .. cached_len[r] + t
 *     ("mini-sglang-learn", request state: extend_len = device_len -
 *     cached_len; autoregression in the deep dive, section 6.1).
 *   - lse_merge: partial results over disjoint token ranges combine by their
 *     log-sum-exp (the split-KV idea named in "mini-sglang-learn", attention
 *     backends passage); used here only as a definition to check against.
 *   - GQA: query head h reads KV head h / (H_q / H_kv) (contiguous groups;
 *     the pages name GQA but give no mapping, so this is the plain reading).
 *   - rope: rotary position embedding of q and k by a cached cos/sin table
 *     (deep dive, section 7.3), the step just before store_kv in each layer.
 *
 * Numbers: inputs are bf16 bit patterns, widened exactly to double; all
 * arithmetic is double; outputs are double.  A NaN anywhere in a gathered row
 * makes the result NaN (no masking), so reads of poisoned rows are visible.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 is the top half of an IEEE binary32; widening is exact. */
static double widen(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---------------------------------------------------------------------- */
/* store_kv                                                                */
/* ---------------------------------------------------------------------- */
/* Rows are row_elems bf16 values.  Token i's row sits at k + i*tok_stride;
 * pool row p at k_pool + p*pool_row_stride.  Tokens are applied in index
 * order.  Returns -1 if an out_loc entry lies outside [0, num_rows). */
int oracle_store_kv(uint16_t *k_pool, uint16_t *v_pool, int64_t pool_row_stride, int64_t num_rows,
                    const uint16_t *k, const uint16_t *v, int64_t tok_stride,
                    const int32_t *out_loc, int64_t n_tokens, int64_t row_elems)
{
    for (int64_t i = 0; i < n_tokens; i++) {
        int64_t row = out_loc[i];
        if (row < 0 || row >= num_rows)
            return -1;
        memcpy(k_pool + row * pool_row_stride, k + i * tok_stride, (size_t)row_elems * 2);
        memcpy(v_pool + row * pool_row_stride, v + i * tok_stride, (size_t)row_elems * 2);
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* one query over one request's logical tokens [j0, j1)                    */
/* ---------------------------------------------------------------------- */
struct pool_view {
    const uint16_t *k_pool, *v_pool; /* layer base of K and V */
    int64_t row_stride;              /* elements between consecutive physical rows */
    int64_t num_rows;
    int num_kv_heads, head_dim;
};

/* scores: scratch of at least (j1 - j0) doubles.  Writes o[head_dim] and *lse.
 * An empty range gives o = 0 and lse = -inf.  Returns -1 on a bad row index. */
static int attend(const struct pool_view *pv, const uint16_t *q, int kv_head, const int32_t *rows,
                  int64_t j0, int64_t j1, double scale, double *scores, double *o, double *lse)
{
    const int d = pv->head_dim;
    for (int c = 0; c < d; c++)
        o[c] = 0.0;
    if (j1 <= j0) {
        *lse = -INFINITY;
        return 0;
    }
    /* scores and their maximum */
    double m = -INFINITY;
    for (int64_t j = j0; j < j1; j++) {
        int64_t row = rows[j];
        if (row < 0 || row >= pv->num_rows)
            return -1;
        const uint16_t *krow = pv->k_pool + row * pv->row_stride + (int64_t)kv_head * d;
        double s = 0.0;
        for (int c = 0; c < d; c++)
            s += widen(q[c]) * widen(krow[c]);
        s *= scale;
        scores[j - j0] = s;
        if (s > m)
            m = s;
    }
    /* unnormalised weights and their sum */
    double l = 0.0;
    for (int64_t j = j0; j < j1; j++) {
        double w = exp(scores[j - j0] - m);
        scores[j - j0] = w;
        l += w;
    }
    /* weighted sum of V rows, then normalise */
    for (int64_t j = j0; j < j1; j++) {
        const uint16_t *vrow = pv->v_pool + (int64_t)rows[j] * pv->row_stride + (int64_t)kv_head * d;
        double w = scores[j - j0];
        for (int c = 0; c < d; c++)
            o[c] += w * widen(vrow[c]);
    }
    for (int c = 0; c < d; c++)
        o[c] = o[c] / l;
    *lse = m + log(l);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* decode                                                                  */
/* ---------------------------------------------------------------------- */
/* q: [batch, num_q_heads, head_dim] bf16.  page_table: [batch, pt_stride].
 * Request r attends over logical tokens [j_begin[r], j_end[r]); j_begin may
 * be NULL (meaning 0), and j_end is the request's seq_len for a full decode.
 * out: [batch, num_q_heads, head_dim]; lse: [batch, num_q_heads] (may be NULL).
 * Returns -1 on bad arguments or a row index outside the pool. */
int oracle_decode(const uint16_t *q, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                  int32_t head_dim, const uint16_t *k_pool, const uint16_t *v_pool,
                  int64_t row_stride, int64_t num_rows, const int32_t *page_table,
                  int64_t pt_stride, const int32_t *j_begin, const int32_t *j_end,
                  double sm_scale, double *out, double *lse)
{
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return -1;
    const int group = num_q_heads / num_kv_heads;
    struct pool_view pv = {k_pool, v_pool, row_stride, num_rows, num_kv_heads, head_dim};
    int64_t longest = 1;
    for (int r = 0; r < batch; r++)
        if (j_end[r] > longest)
            longest = j_end[r];
    double *scores = malloc(sizeof(double) * (size_t)longest);
    if (!scores)
        return -1;
    int rc = 0;
    for (int r = 0; r < batch && rc == 0; r++) {
        const int32_t *rows = page_table + (int64_t)r * pt_stride;
        int64_t j0 = j_begin ? j_begin[r] : 0, j1 = j_end[r];
        if (j1 > pt_stride)
            rc = -1;
        for (int h = 0; h < num_q_heads && rc == 0; h++) {
            const uint16_t *qv = q + ((int64_t)r * num_q_heads + h) * head_dim;
            double dummy_lse;
            rc = attend(&pv, qv, h / group, rows, j0, j1, sm_scale, scores,
                        out + ((int64_t)r * num_q_heads + h) * head_dim,
                        lse ? &lse[(int64_t)r * num_q_heads + h] : &dummy_lse);
        }
    }
    free(scores);
    return rc;
}

/* ---------------------------------------------------------------------- */
/* extend (causal, chunked prefill)                                        */
/* ---------------------------------------------------------------------- */
/* q: [T, num_q_heads, head_dim] bf16, the new tokens of all requests packed in
 * request order (request r's tokens start at the sum of earlier extend_lens).
 * Token t of request r is at absolute position cached_lens[r] + t and attends
 * over logical tokens [0, cached_lens[r] + t + 1).
 * out: [T, num_q_heads, head_dim].  Returns -1 on bad arguments. */
int oracle_extend(const uint16_t *q, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                  int32_t head_dim, const uint16_t *k_pool, const uint16_t *v_pool,
                  int64_t row_stride, int64_t num_rows, const int32_t *page_table,
                  int64_t pt_stride, const int32_t *cached_lens, const int32_t *extend_lens,
                  double sm_scale, double *out)
{
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return -1;
    const int group = num_q_heads / num_kv_heads;
    struct pool_view pv = {k_pool, v_pool, row_stride, num_rows, num_kv_heads, head_dim};
    int64_t longest = 1;
    for (int r = 0; r < batch; r++)
        if (cached_lens[r] + extend_lens[r] > longest)
            longest = cached_lens[r] + extend_lens[r];
    double *scores = malloc(sizeof(double) * (size_t)longest);
    if (!scores)
        return -1;
    int rc = 0;
    int64_t tok = 0; /* packed index of request r's first new token */
    for (int r = 0; r < batch && rc == 0; r++) {
        const int32_t *rows = page_table + (int64_t)r * pt_stride;
        if (cached_lens[r] + extend_lens[r] > pt_stride)
            rc = -1;
        for (int t = 0; t < extend_lens[r] && rc == 0; t++) {
            int64_t visible = (int64_t)cached_lens[r] + t + 1;
            for (int h = 0; h < num_q_heads && rc == 0; h++) {
                int64_t at = ((tok + t) * num_q_heads + h) * head_dim;
                double unused_lse;
                rc = attend(&pv, q + at, h / group, rows, 0, visible, sm_scale, scores,
                            out + at, &unused_lse);
            }
        }
        tok += extend_lens[r];
    }
    free(scores);
    return rc;
}

/* ---------------------------------------------------------------------- */
/* log-sum-exp merge of partial results                                    */
/* ---------------------------------------------------------------------- */
/* o_parts: [n_parts, n_vec, head_dim]; lse_parts: [n_parts, n_vec].  For each
 * vector, parts with lse = -inf (empty ranges) carry no weight; if every part
 * is empty the result is o = 0, lse = -inf. */
void oracle_lse_merge(int64_t n_parts, int64_t n_vec, int32_t head_dim, const double *o_parts,
                      const double *lse_parts, double *out, double *lse_out)
{
    for (int64_t i = 0; i < n_vec; i++) {
        double top = -INFINITY;
        for (int64_t s = 0; s < n_parts; s++)
            if (lse_parts[s * n_vec + i] > top)
                top = lse_parts[s * n_vec + i];
        double *o = out + i * head_dim;
        for (int c = 0; c < head_dim; c++)
            o[c] = 0.0;
        if (top == -INFINITY) {
            if (lse_out)
                lse_out[i] = -INFINITY;
            continue;
        }
        double total = 0.0;
        for (int64_t s = 0; s < n_parts; s++) {
            double ls = lse_parts[s * n_vec + i];
            if (ls == -INFINITY)
                continue;
            double w = exp(ls - top);
            total += w;
            const double *os = o_parts + (s * n_vec + i) * head_dim;
            for (int c = 0; c < head_dim; c++)
                o[c] += w * os[c];
        }
        for (int c = 0; c < head_dim; c++)
            o[c] = o[c] / total;
        if (lse_out)
            lse_out[i] = top + log(total);
    }
}

/* ---------------------------------------------------------------------- */
/* rotary position embedding (RoPE)                                        */
/* ---------------------------------------------------------------------- */
/* "mini-sglang architecture deep dive", section 7.3 (RoPE): a cache holds,
 * for every position p, the row [cos(p*f_0) .. cos(p*f_{d/2-1}),
 * sin(p*f_0) .. sin(p*f_{d/2-1})] in float32, with f_i = base^(-2i/d) and
 * rotary_dim = head_size = d; the library call it makes rotates q and k in
 * place by the cached angles of each token's position.  The pages do not say
 * which elements form a rotated pair; this follows the half-split pairing
 * (element i with element i + d/2), the default of the routine the page
 * calls:
 *     y[i]       = x[i] * cos_i - x[i + d/2] * sin_i
 *     y[i + d/2] = x[i + d/2] * cos_i + x[i] * sin_i,      i < d/2.
 * x: [n_tokens, num_heads, head_dim] bf16 bits (token stride
 * num_heads*head_dim); cos_sin_cache: [max_positions, head_dim] float32;
 * out: [n_tokens, num_heads, head_dim] double.  Returns -1 if a position lies
 * outside [0, max_positions) or head_dim is odd. */
int oracle_rope(const uint16_t *x, int64_t n_tokens, int32_t num_heads, int32_t head_dim,
                const int32_t *positions, const float *cos_sin_cache, int64_t max_positions,
                double *out)
{
    if (head_dim % 2 != 0)
        return -1;
    const int32_t half = head_dim / 2;
    for (int64_t i = 0; i < n_tokens; i++) {
        const int64_t pos = positions[i];
        if (pos < 0 || pos >= max_positions)
            return -1;
        const float *cs = cos_sin_cache + pos * head_dim;
        for (int32_t h = 0; h < num_heads; h++) {
            const int64_t at = (i * num_heads + h) * (int64_t)head_dim;
            for (int32_t j = 0; j < half; j++) {
                const double c = (double)cs[j], s = (double)cs[half + j];
                const double x1 = widen(x[at + j]), x2 = widen(x[at + half + j]);
                out[at + j] = x1 * c - x2 * s;
                out[at + half + j] = x2 * c + x1 * s;
            }
        }
    }
    return 0;
}
