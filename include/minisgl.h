/*
 * minisgl.h -- C ABI of the GB300 (sm_103a) paged KV-pool attention library.
 *
 * Three operations make up the attention step of a serving engine that keeps
 * its KV cache in one paged pool (the mini-sglang design):
 *
 *   minisgl_store_kv     scatter this step's new K/V token rows into the pool
 *   minisgl_decode_attn  one query token per request, split-KV, then an LSE merge
 *   minisgl_store_decode_attn  store_kv and decode in one pass
 *   minisgl_extend_attn  causal attention for the new tokens of chunked prefill
 *   minisgl_rope_store_kv  rotary position embedding of q and k fused with store_kv
 *   minisgl_cascade_decode_attn  decode for requests sharing a prefix, prefix read once
 *   minisgl_cascade_extend_attn  extend for requests sharing a prefix, prefix pass + own rows
 *
 * Sources of the definitions (page title, section):
 *   [deep-dive]  "mini-sglang 架构深度解读" (mini-sglang architecture deep dive,
 *                tinymind.me): section 6.2 MHAKVCache layout, section 3.6
 *                page-table figure, section 5 attention backends.
 *   [learn]      "doc-mini-sglang-learn" (mini-sglang learning notes): the
 *                paged KV pool chapter (pool shape, store_kv, dummy page,
 *                page_table alignment, page_size), the request-state passage
 *                (cached_len / extend_len), the chunked-prefill chapter and
 *                the attention-backend chapter (FlashDecoding-style split-KV).
 *   [sglang]     "SGLang 源码导读" (SGLang source reading guide): ForwardBatch
 *                fields seq_lens, extend_prefix_lens, extend_seq_lens,
 *                out_cache_loc.
 *
 * Conventions for every entry point
 *   - All tensor arguments are DEVICE pointers owned by the caller; the
 *     library never allocates or frees device memory at run time.  Besides a
 *     thread-local error string it keeps only two things in its own,
 *     statically sized device memory: the 32 MiB scratch array of
 *     minisgl_decode_attn_noalloc, and 64 work-ticket counters that
 *     minisgl_extend_attn uses to hand out work items to its thread blocks
 *     when the caller passes no counter of its own (each such call draws one
 *     of the 64 in turn and leaves it at zero when its kernel completes, so
 *     more than 64 such calls in flight at the same time on unordered
 *     streams would share counters and give wrong results; callers that run
 *     extend calls concurrently pass their own counters).  Per device it
 *     also creates, on first use, one CUDA stream and two events that
 *     minisgl_cascade_decode_attn uses to run its two parts side by side.
 *   - Element type is bf16 for K, V, Q and the output (MINISGL_BF16); index
 *     tensors are int32.  Strides are in elements.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  No call synchronises with the host.  minisgl_store_decode_attn,
 *     minisgl_extend_attn (with minisgl_store_kv; with and without a caller
 *     work counter), minisgl_cascade_decode_attn (including its fork onto the
 *     library's second stream and the join back) and
 *     minisgl_cascade_extend_attn are tested captured in a CUDA graph and
 *     replayed, with their pointers fixed; the first cascade-decode call on a
 *     device creates that stream and its events, so make it before capture.
 *   - Return value: MINISGL_OK, or a negative MINISGL_ERR_* code with a
 *     message available from minisgl_last_error().  Argument checks happen on
 *     the host before any launch; a launch failure returns MINISGL_ERR_CUDA.
 *   - Kernels never trap.  Index VALUES live on the device and are not checked
 *     by the host: a page_table / out_loc entry outside [0, num_rows) is a
 *     caller error; the kernels clamp it into the pool so that no access
 *     leaves the caller's buffers, and the affected results are unspecified.
 *     seq_lens / cached_lens + extend_lens larger than the page_table width
 *     are likewise clamped to the width.
 *   - Alignment: pool bases, k/v/q/out bases and all row strides must give
 *     16-byte aligned rows (bases 16-byte aligned, strides multiples of 8
 *     elements).
 */
#ifndef MINISGL_H
#define MINISGL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    MINISGL_OK = 0,
    MINISGL_ERR_ARG = -1,         /* null pointer, negative size, bad layer */
    MINISGL_ERR_DTYPE = -2,       /* pool dtype is not MINISGL_BF16 */
    MINISGL_ERR_SHAPE = -3,       /* head counts / strides / alignment inconsistent */
    MINISGL_ERR_UNSUPPORTED = -4, /* head_dim or group size this build has no kernel for */
    MINISGL_ERR_CUDA = -5,        /* a CUDA call or kernel launch failed */
    MINISGL_ERR_WORKSPACE = -6    /* workspace missing or too small */
};

enum { MINISGL_BF16 = 1 };

/*
 * The KV pool [deep-dive 6.2; learn, paged KV pool]: logically
 * (2, L, R, H_kv, d) -- K/V, layer, physical token row, KV head, head dim.
 * Per layer, K and V are each an (R, H_kv, d) array of token rows and a
 * token's physical position is its row number.  page_size s only describes
 * how rows were allocated (R = P * s); the kernels never assume pages are
 * contiguous, because page_table entries are raw rows.
 *   element (kv, l, row, h, c) of K is at  k_base + l*layer_stride + row*row_stride + h*head_dim + c
 * LayerFirst allocation gives layer_stride = R*H_kv*d and row_stride = H_kv*d;
 * PageFirst (pages outermost) gives layer_stride = H_kv*d and
 * row_stride = L*H_kv*d.  Both are accepted.
 */
typedef struct {
    void *k_base;          /* device: K of layer 0, row 0 */
    void *v_base;          /* device: V of layer 0, row 0 */
    int64_t layer_stride;  /* elements between layers */
    int64_t row_stride;    /* elements between physical rows; >= num_kv_heads*head_dim */
    int32_t num_layers;
    int32_t num_rows;      /* R, including any dummy page rows */
    int32_t num_kv_heads;  /* H_kv local to this GPU */
    int32_t head_dim;      /* d: 64 or 128 */
    int32_t page_size;     /* s: informational (1, 16, 32, 64 ...) */
    int32_t dtype;         /* MINISGL_BF16 */
} minisgl_kv_pool;

/*
 * store_kv [learn, paged KV pool: "store_kv" passage; deep-dive 6.2].
 * For i < n_tokens and every KV head h and channel c:
 *     K[layer][out_loc[i]][h][c] = k[i*k_tok_stride + h*head_dim + c]
 *     V[layer][out_loc[i]][h][c] = v[i*v_tok_stride + h*head_dim + c]
 * k, v: device bf16, one row of num_kv_heads*head_dim elements per token.
 * out_loc: device int32 [n_tokens], physical rows.  Bit-exact copy.  Tokens
 * that share a row (CUDA-Graph padding requests all write the dummy row)
 * race; the row ends up holding one of their values, so callers give such
 * tokens identical k/v.  n_tokens == 0 is a no-op.
 */
int minisgl_store_kv(const minisgl_kv_pool *pool, int32_t layer, const void *k, const void *v,
                     int64_t k_tok_stride, int64_t v_tok_stride, const int32_t *out_loc,
                     int32_t n_tokens, void *stream);

/*
 * Workspace size for minisgl_decode_attn, in bytes, for up to `max_splits`
 * partial results per (request, KV head) (2 <= max_splits <= 256; 16 is a
 * good default).  Layout of a workspace of this size, for the record (the
 * caller does not need to read it):
 *   int32 split_count[batch * num_kv_heads]            (at offset 0, padded to 256 B)
 *   float lse[batch * num_q_heads * max_splits]        natural-log LSE per partial
 *   float o[batch * num_q_heads * max_splits * head_dim] normalised partial outputs
 * Index of partial s of request r, query head h: (r*num_q_heads + h)*max_splits + s.
 */
size_t minisgl_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t max_splits);

/*
 * Decode attention [learn, paged KV pool and attention-backend chapters;
 * deep-dive 5.3 PagedAttention].  For request r < batch, query head
 * h < num_q_heads, KV head g = h / (num_q_heads / num_kv_heads) (GQA, contiguous
 * groups), and n = seq_lens[r] (the context INCLUDING the token stored this
 * step by minisgl_store_kv):
 *     S_j = sm_scale * <q[r,h,:], K[layer][page_table[r*pt_row_stride + j]][g][:]>,  j < n
 *     out[r,h,:] = sum_j softmax(S)_j * V[layer][page_table[r*pt_row_stride + j]][g][:]
 * q: device bf16 [batch, num_q_heads, head_dim] contiguous.
 * page_table: device int32, row r at page_table + r*pt_row_stride, raw
 *   physical rows; columns j >= seq_lens[r] are never read.
 * seq_lens: device int32 [batch].  n == 0 gives out = 0.
 * out: device bf16 [batch, num_q_heads, head_dim] contiguous.
 * workspace: device, caller-owned, at least
 *   minisgl_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, 2)
 *   bytes; the number of splits the kernel may use grows with its size.
 * split_tokens: 0 lets the kernel balance the KV length over all SMs (the
 *   normal setting); a positive value asks for about that many tokens per
 *   partial result (rounded up to 16, and raised if the workspace is too
 *   small for it) -- used to test the merge at chosen split counts.
 * Launches a split-KV partial kernel and, when any request was split, the
 * log-sum-exp merge kernel, both on `stream`.
 * Supported: head_dim in {64, 128}; 1 <= num_q_heads/num_kv_heads <= 16;
 * batch <= 4096.
 */
int minisgl_decode_attn(const minisgl_kv_pool *pool, int32_t layer, const void *q,
                        int32_t num_q_heads, const int32_t *page_table, int32_t batch,
                        int64_t pt_row_stride, int32_t pt_width, const int32_t *seq_lens,
                        float sm_scale, void *out, void *workspace, size_t workspace_bytes,
                        int32_t split_tokens, void *stream);

/*
 * store_kv fused into decode [learn, paged KV pool: each layer stores the
 * step's new K/V rows, then attends].  Same results as minisgl_store_kv of
 * (k, v, out_loc) followed by minisgl_decode_attn with the remaining
 * arguments, in one kernel pass: the warp that reads a request's last tile
 * writes the request's new K/V rows (one per request: k[r], v[r], token
 * strides in elements) to row out_loc[r], and positions whose page-table row
 * is the request's out_loc row read the new rows directly.  Conditions (the
 * decode step satisfies them): every seq_lens[r] >= 1, and no request reads
 * another request's out_loc row unless both store identical values there
 * (CUDA-Graph padding requests sharing the dummy row).  Rows of requests
 * with seq_lens[r] == 0 are not stored.
 */
int minisgl_store_decode_attn(const minisgl_kv_pool *pool, int32_t layer, const void *k,
                              const void *v, int64_t k_tok_stride, int64_t v_tok_stride,
                              const int32_t *out_loc, const void *q, int32_t num_q_heads,
                              const int32_t *page_table, int32_t batch, int64_t pt_row_stride,
                              int32_t pt_width, const int32_t *seq_lens, float sm_scale, void *out,
                              void *workspace, size_t workspace_bytes, int32_t split_tokens,
                              void *stream);

/*
 * Extend (chunked-prefill) attention [learn: request-state passage
 * extend_len = device_len - cached_len, chunked-prefill chapter; sglang:
 * ForwardBatch extend_prefix_lens / extend_seq_lens].  Request r has
 * C = cached_lens[r] tokens already in the pool and E = extend_lens[r] new
 * tokens, whose K/V the caller has already stored (minisgl_store_kv) at the
 * rows page_table[r, C .. C+E-1].  New token t (0 <= t < E) is at absolute
 * position C + t and attends causally to logical tokens 0 .. C + t:
 *     out[q_offsets[r]+t, h, :] = sum_{j <= C+t} softmax_j(sm_scale * <q[q_offsets[r]+t,h,:], K_j[g]>) V_j[g]
 * q: device bf16 [total_q_tokens, num_q_heads, head_dim] packed in request order.
 * q_offsets: device int32 [batch+1], exclusive prefix sum of extend_lens
 *   (q_offsets[batch] == total_q_tokens).
 * cached_lens, extend_lens: device int32 [batch].
 * page_table: as for decode; pt_width columns per row.
 * out: device bf16 [total_q_tokens, num_q_heads, head_dim].
 * sm_scale must be positive and finite (MINISGL_ERR_ARG otherwise).
 * work_counter: optional device uint32[2], 8-byte aligned, zero before its
 *   first use; the kernel hands out work items to its thread blocks from it
 *   and leaves it at zero when it completes.  Calls that may run at the same
 *   time (unordered streams) need different counters; calls ordered on one
 *   stream may share one.  NULL: one of the library's 64 slots (see above).
 * Runs on the tensor cores (tcgen05, accumulators in tensor memory).
 * Supported: head_dim 64 or 128; num_q_heads/num_kv_heads any of 1..16;
 * batch <= 4096.
 */
int minisgl_extend_attn(const minisgl_kv_pool *pool, int32_t layer, const void *q,
                        int32_t num_q_heads, const int32_t *page_table, int32_t batch,
                        int64_t pt_row_stride, int32_t pt_width, const int32_t *cached_lens,
                        const int32_t *extend_lens, const int32_t *q_offsets,
                        int32_t total_q_tokens, float sm_scale, void *out, uint32_t *work_counter,
                        void *stream);

/*
 * Workspace size, in bytes, for minisgl_cascade_decode_attn with this batch
 * and head shape; 0 for invalid sizes.  The number of prefix chunks a call
 * may use (up to 32) grows with the SM count of the CURRENT device, so query
 * the size with the device current that will run the call: a workspace sized
 * on a device with fewer SMs can be too small for one with more (the call
 * then fails with MINISGL_ERR_WORKSPACE).
 */
size_t minisgl_cascade_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim);

/*
 * Decode attention for a batch whose requests share a cached prefix
 * [learn, radix-cache chapter: requests matching a cached prefix point at its
 * rows; deep-dive 5.3 PagedAttention].  Same definition and arguments as
 * minisgl_decode_attn, plus shared_len = P: the caller guarantees that the
 * first P page-table entries are the same physical rows in every row of the
 * batch and that every seq_lens[r] >= P (results are unspecified otherwise;
 * the call checks nothing on the device; minisgl_check_shared_prefix counts
 * violations in a debugging run).  The shared rows are read once per KV
 * head for the whole batch instead of once per request: the P prefix
 * positions are attended by all B*G query rows of a KV head at once on the
 * tensor cores (in chunks spread over the SMs), each request's own positions
 * [P, seq_len) by the split-KV decode partial kernel, and the parts are
 * merged by their log-sum-exp in fp32.  When the prefix part leaves at
 * least 24 SMs free, the suffix part runs on those SMs at the same time, on
 * a library-owned second stream forked from `stream` and joined back to it
 * with events (so the call stays capturable in a CUDA graph); otherwise the
 * parts run one after the other on `stream`.  The library's second stream
 * is shared by all calls on a device, so two cascade calls on different
 * caller streams serialise their suffix parts.
 * workspace: device, 256-byte aligned, at least
 *   minisgl_cascade_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim)
 *   bytes.  Its first 256 bytes hold a work counter that must be zero before
 *   the workspace's first use (every call leaves it at zero); calls that may
 *   run at the same time need different workspaces.
 * Cascade pays when the shared prefix dominates the batch's bytes; with
 * short prefixes its fixed costs (three kernels, the fp32 partials) exceed
 * the re-read it saves and plain minisgl_decode_attn is faster (measured on
 * 64 requests of 16 query / 8 KV heads: plain decode faster at a 256-token
 * prefix, cascade 1.36x faster at 1024 and 3.2x at 4096).
 * Supported: head_dim 64 or 128; num_q_heads/num_kv_heads any of 1..16;
 * 1 <= shared_len <= pt_width; batch <= 4096.
 */
int minisgl_cascade_decode_attn(const minisgl_kv_pool *pool, int32_t layer, const void *q,
                                int32_t num_q_heads, const int32_t *page_table, int32_t batch,
                                int64_t pt_row_stride, int32_t pt_width, const int32_t *seq_lens,
                                int32_t shared_len, float sm_scale, void *out, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * Workspace size, in bytes, for minisgl_cascade_extend_attn (an fp32 partial
 * output row and LSE per new token and query head, and a work counter); 0
 * for invalid sizes.
 */
size_t minisgl_cascade_extend_workspace_bytes(int32_t total_q_tokens, int32_t num_q_heads,
                                              int32_t head_dim);

/*
 * Extend attention for a chunked-prefill batch whose requests share a cached
 * prefix [learn, radix-cache chapter; chunked-prefill chapter; request-state
 * passage].  Same definition, arguments and result as minisgl_extend_attn,
 * plus shared_len = P: the caller guarantees that the first P page-table
 * entries are the same physical rows in every row of the batch and that
 * every cached_lens[r] >= P (results are unspecified otherwise; the call
 * checks nothing on the device; minisgl_check_shared_prefix counts
 * violations).  Two tensor-core passes: (1) every new token of the
 * batch against the P shared positions as one block, read once per KV head,
 * leaving fp32 partial rows and LSEs in the workspace; (2) each request's own
 * positions P .. C+t causally, with the partial from (1) folded in by
 * log-sum-exp before the bf16 output is written.
 * workspace: device, 256-byte aligned, at least
 *   minisgl_cascade_extend_workspace_bytes(total_q_tokens, num_q_heads, head_dim)
 *   bytes; its first 256 bytes hold a work counter that must be zero before
 *   the workspace's first use (every call leaves it at zero); calls that may
 *   run at the same time need different workspaces.
 * The new tokens' scores against the shared positions are computed exactly
 * as often as in minisgl_extend_attn (every token sees every shared
 * position), so the work is the same; the benefit is the shared K/V tiles
 * being gathered once per block of 2*floor(128/G) tokens of the whole batch,
 * at the price of the fp32 partial written and read back (8*d + 8 bytes per
 * token and query head).
 * Supported: as minisgl_extend_attn; 1 <= shared_len <= pt_width.
 */
int minisgl_cascade_extend_attn(const minisgl_kv_pool *pool, int32_t layer, const void *q,
                                int32_t num_q_heads, const int32_t *page_table, int32_t batch,
                                int64_t pt_row_stride, int32_t pt_width, const int32_t *cached_lens,
                                const int32_t *extend_lens, const int32_t *q_offsets,
                                int32_t total_q_tokens, int32_t shared_len, float sm_scale, void *out,
                                void *workspace, size_t workspace_bytes, void *stream);

/*
 * Rotary position embedding fused with store_kv [deep-dive 7.3 RoPE: a
 * float32 [cos | sin] table per position, rotary_dim = head_dim, q and k
 * rotated in place by each token's position; learn, paged KV pool: store_kv
 * then scatters the new K/V rows].  For token i < n_tokens at position
 * p = positions[i], every head x of q and of k is rotated pairwise, element j
 * with element j + d/2 (the half-split pairing; the pages name the library
 * call but not the pairing):
 *     y[j]       = x[j] * cos_j(p) - x[j + d/2] * sin_j(p)
 *     y[j + d/2] = x[j + d/2] * cos_j(p) + x[j] * sin_j(p),     j < d/2,
 * with cos_j(p) = cos_sin_cache[p*d + j], sin_j(p) = cos_sin_cache[p*d + d/2 + j].
 * Arithmetic in fp32 from the bf16 inputs, results rounded to nearest bf16.
 *   q: device bf16, token i's heads at q + i*q_tok_stride, [num_q_heads, d];
 *      overwritten with the rotated q.
 *   k, v: device bf16 [n_tokens, H_kv, d] rows (token strides in elements);
 *      read only.  The rotated k is written to K[layer][out_loc[i]] and v to
 *      V[layer][out_loc[i]] (v bit-exact); k itself is not rotated in place.
 *   positions, out_loc: device int32 [n_tokens].
 *   cos_sin_cache: device float32 [max_positions, d], 16-byte aligned.
 * Positions outside [0, max_positions) and rows outside [0, num_rows) are a
 * caller error: they are clamped into range (results unspecified), never
 * trapped.  Tokens sharing a row (CUDA-Graph padding) race as in
 * minisgl_store_kv; give them identical k, v and positions.
 * head_dim 64 or 128.  n_tokens == 0 is a no-op.
 */
int minisgl_rope_store_kv(const minisgl_kv_pool *pool, int32_t layer, void *q, int32_t num_q_heads,
                          int64_t q_tok_stride, const void *k, const void *v, int64_t k_tok_stride,
                          int64_t v_tok_stride, const int32_t *positions, const float *cos_sin_cache,
                          int32_t max_positions, const int32_t *out_loc, int32_t n_tokens,
                          void *stream);

/*
 * Decode attention that allocates nothing (no counterpart in the pages; this
 * is a convenience of this library).  Same arguments and results as
 * minisgl_decode_attn minus the workspace: the split-KV scratch comes from a
 * 32 MiB array in the library's own device memory instead of from the caller.
 * For callers that cannot allocate device memory at run time -- an engine that
 * has already given nearly all free HBM to its KV pool, code inside a host
 * application that owns the device allocator, or a decode loop that cannot
 * afford cudaMalloc/cudaFree synchronising the device.
 *   - Every GPU on which the library is loaded holds the 32 MiB array until the
 *     process exits.
 *   - Every call looks up the array's device address on the current device
 *     with cudaGetSymbolAddress (a host-side lookup, never cached, so a
 *     device reset cannot leave a stale address behind).  The first call on
 *     each device also loads the library's module there: make that first
 *     call before any stream capture.
 *   - Sizes whose scratch (minisgl_decode_workspace_bytes(..., 2)) exceeds
 *     32 MiB are rejected with MINISGL_ERR_WORKSPACE and a message: at
 *     head_dim 128 that is about batch * num_q_heads > 32,500 (for example
 *     16 query heads over 8 KV heads: batch 2028 fits, 2029 does not), at
 *     head_dim 64 about batch * num_q_heads > 64,000.
 *   - All calls share the array: calls whose kernels can overlap on the GPU
 *     (unordered streams) race and give wrong results.  Nothing in the array
 *     needs to start at zero; every value a call reads, it wrote first.
 */
int minisgl_decode_attn_noalloc(const minisgl_kv_pool *pool, int32_t layer, const void *q,
                                int32_t num_q_heads, const int32_t *page_table, int32_t batch,
                                int64_t pt_row_stride, int32_t pt_width, const int32_t *seq_lens,
                                float sm_scale, void *out, int32_t split_tokens, void *stream);

/*
 * Index check: a debugging aid with no counterpart in the pages, for callers
 * who want to know whether their index tensors address rows outside the pool
 * (the calls above never check index values on the device; they clamp them,
 * with unspecified results).  It reads exactly the entries a decode or
 * extend call over the same tensors would read and counts, on the device:
 *   counts[0]: page_table[r, j] outside [0, num_rows), r < batch,
 *              j < min(max(lens[r], 0), pt_width);
 *   counts[1]: out_loc[i] outside [0, num_rows), i < n_out;
 *   counts[2]: lens[r] outside [0, pt_width].
 * The page_table rows are [learn, paged KV pool: page_table alignment
 * passage] raw physical rows padded to pt_width; entries past a request's
 * length are not read.
 *   page_table: device int32, row r at page_table + r*pt_row_stride.
 *   lens: device int32 [batch], the page-table positions each request reads
 *      (seq_lens for decode; cached_lens + extend_lens for extend).
 *   out_loc: device int32 [n_out] (may be NULL when n_out == 0).
 *   counts: device uint32 [3], overwritten (zeroed on `stream`, then
 *      counted); read them after the stream, e.g. with a copy to the host.
 * No kernel traps or synchronises with the host.  batch == 0 and n_out == 0
 * just zero the counts.
 */
int minisgl_check_indices(const int32_t *page_table, int32_t batch, int64_t pt_row_stride,
                          int32_t pt_width, const int32_t *lens, const int32_t *out_loc,
                          int32_t n_out, int32_t num_rows, uint32_t *counts, void *stream);

/*
 * Shared-prefix check: a debugging aid with no counterpart in the pages, for
 * callers of minisgl_cascade_decode_attn / minisgl_cascade_extend_attn, which
 * trust (and never check) that the first shared_len page-table entries are
 * the same physical rows in every request [learn, radix-cache chapter] and
 * that every request reads at least shared_len positions.  Counts on the
 * device:
 *   counts[0]: entries page_table[r, j] != page_table[0, j], 0 < r < batch,
 *              j < shared_len;
 *   counts[1]: requests with lens[r] < shared_len (lens: seq_lens for
 *              decode, cached_lens for extend).
 *   counts: device uint32 [2], overwritten (zeroed on `stream`, then counted).
 * 1 <= shared_len <= pt_width.  No kernel traps or synchronises with the host.
 */
int minisgl_check_shared_prefix(const int32_t *page_table, int32_t batch, int64_t pt_row_stride,
                                int32_t pt_width, int32_t shared_len, const int32_t *lens,
                                uint32_t *counts, void *stream);

/* Message of the last error on the calling thread ("" if none). */
const char *minisgl_last_error(void);

/* Number of streaming multiprocessors of the current device (0 on error);
 * the persistent kernels size their grids from it. */
int32_t minisgl_device_sm_count(void);

/* Debugging and measurement aid: turn programmatic dependent launch on (1)
 * or off (0) for every later launch of this library in the process, and
 * return the previous setting.  With it on (the default, unless the
 * environment held MINISGL_PDL=0 when the first launch was made) each kernel
 * may be launched while the previous kernel in its stream is finishing and
 * waits on the device for that kernel's results (griddepcontrol.wait); with
 * it off every launch waits for the previous kernel to complete.  Results
 * are the same either way; only the time between kernels changes.  Not
 * thread-safe with respect to launches already being set up on other host
 * threads. */
int minisgl_debug_set_pdl(int enabled);

/* Debugging aid: how many bounded waits inside the tensor-core kernels ran
 * out of time since the library was loaded on the current device.  A
 * non-zero count means some minisgl_extend_attn output is garbage.  This call
 * synchronises with the device (it reads a device counter), so it is not
 * for the hot path. */
int minisgl_debug_timeout_count(uint32_t *count);

#ifdef __cplusplus
}
#endif

#endif /* MINISGL_H */
