// kernels.h -- host-side launch interface between the C ABI (abi.cu) and the
// kernel translation units.  Internal to the library.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace minisgl {

// Whether launches carry the programmatic-stream-serialization attribute
// (on unless the environment holds MINISGL_PDL=0 when the library loads, or
// minisgl_debug_set_pdl turned it off).  Kernels call griddepcontrol.wait
// either way; without the attribute it returns at once because the launch
// already waited for the previous kernel.
bool pdl_enabled();

// Launch with programmatic stream serialization, so this kernel's launch and
// prologue overlap the tail of the previous kernel in the stream; the kernel
// itself calls griddepcontrol.wait before touching global memory.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

struct StoreArgs {
    void *k_layer, *v_layer;      // layer base of K / V in the pool
    int64_t row_stride;           // elements between pool rows
    int32_t num_rows;
    const void *k, *v;            // new rows
    int64_t k_tok_stride, v_tok_stride;
    const int32_t *out_loc;
    int32_t n_tokens;
    int32_t row_elems;            // num_kv_heads * head_dim
};
cudaError_t launch_store_kv(const StoreArgs &a, cudaStream_t s);

struct DecodeArgs {
    const void *q;                // [B, Hq, D]
    const void *k_layer, *v_layer;
    int64_t row_stride;
    int32_t num_rows;
    const int32_t *page_table;
    int64_t pt_stride;
    int32_t pt_width;
    const int32_t *seq_lens;
    int32_t batch, num_q_heads, num_kv_heads, head_dim;
    float sm_scale;
    void *out;                    // [B, Hq, D] bf16
    int32_t *split_count;         // workspace parts
    float *ws_lse, *ws_o;
    int32_t max_splits;
    int32_t split_tokens;         // 0 = automatic
    float *lse_out;               // optional [B, Hq] natural-log LSE of each output row
    // optional fused store_kv: request r's new K/V rows (k_new + r*new_k_stride,
    // v_new + r*new_v_stride) go to pool row out_loc[r]; null out_loc = no store
    const int32_t *out_loc;
    const void *k_new, *v_new;
    int64_t new_k_stride, new_v_stride;
    // request r's context is seq_lens[r] - len_offset positions of its
    // page_table row (the cascade suffix: the row pointer is already moved
    // past the shared prefix)
    int32_t len_offset = 0;
    // 1: every stream, whole or split, leaves fp32 partials and LSEs in the
    // workspace (split 0 for a whole stream) and no merge kernel runs
    int32_t partials_only = 0;
    // > 0: a grid for at most this many SMs (the rest of the GPU runs other work)
    int32_t max_sms = 0;
};
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s);

struct ExtendArgs {
    const void *q;                // [T, Hq, D]
    const void *k_layer, *v_layer;
    int64_t row_stride;
    int32_t num_rows;
    const int32_t *page_table;
    int64_t pt_stride;
    int32_t pt_width;
    const int32_t *cached_lens, *extend_lens, *q_offsets;
    int32_t batch, total_q_tokens, num_q_heads, num_kv_heads, head_dim;
    float sm_scale;
    void *out;                    // [T, Hq, D] bf16 (unused when out_f32 is set)
    int32_t prefix_only;          // 1: every new token sees exactly its C cached positions
    float *out_f32;               // optional [T, Hq, D] fp32 normalised output
    float *lse_out;               // [T, Hq] natural-log LSE, with out_f32
    const int32_t *out_offsets;   // optional [B]: first output row of each request (else q_offsets)
    // Prefix chunks of a shared-prefix decode (with prefix_only): request c is
    // chunk c of the prefix_len shared positions, prefix_chunk_len long (the
    // last may be shorter), its page-table row at page_table + c*pt_stride;
    // each chunk reads q rows 0 .. prefix_queries-1 and writes output rows
    // c*prefix_queries ..  The length arrays are not read.  0 = off.
    int32_t prefix_chunk_len = 0, prefix_len = 0, prefix_queries = 0;
    // optional work-ticket counter (2 x uint32, zero before first use, left at
    // zero); null = one of the library's 64 slots, taken in turn
    unsigned int *sched = nullptr;
    // request r has cached_lens[r] - len_offset cached positions in its
    // page-table row (the cascade suffix: the row pointer is already moved
    // past the shared prefix)
    int32_t len_offset = 0;
    // optional fp32 partial result of the same output rows over other
    // positions ([T, Hq, D] normalised rows and [T, Hq] natural-log LSEs,
    // indexed like out): folded into the bf16 output by log-sum-exp
    const float *merge_o = nullptr, *merge_lse = nullptr;
};
cudaError_t launch_extend(const ExtendArgs &a, cudaStream_t s);
// CTAs launch_extend will use for these arguments
int extend_grid(const ExtendArgs &a);

// Shared-prefix (cascade) decode: the prefix part's fp32 partials (written by
// the extend kernel in prefix-chunk mode), the suffix decode (partials only)
// and the merge of both.
struct CascadeArgs {
    const int32_t *seq_lens;      // [B]
    int32_t batch, num_q_heads, head_dim;
    int32_t shared_len, chunks;
    float *pre_o, *pre_lse;       // [chunks, B, Hq, D], [chunks, B, Hq]
    DecodeArgs suffix;            // the suffix decode (workspace parts filled in by the caller)
    void *out;                    // [B, Hq, D] bf16
};
// prefix: the extend launch over the prefix chunks (prefix-chunk mode)
cudaError_t launch_cascade(const CascadeArgs &c, const ExtendArgs &prefix, cudaStream_t s);

struct RopeStoreArgs {
    void *k_layer, *v_layer;      // layer base of K / V in the pool
    int64_t row_stride;           // elements between pool rows
    int32_t num_rows;
    void *q;                      // [N, H_q, D], rotated in place
    int64_t q_tok_stride;
    const void *k, *v;            // new rows [N, H_kv, D]
    int64_t k_tok_stride, v_tok_stride;
    const int32_t *positions;     // [N]
    const float *cos_sin;         // [max_positions, D]: cos | sin
    int32_t max_positions;
    const int32_t *out_loc;       // [N]
    int32_t n_tokens, num_q_heads, num_kv_heads, head_dim;
};
cudaError_t launch_rope_store_kv(const RopeStoreArgs &a, cudaStream_t s);

// Count index values outside the pool (a debugging aid; see minisgl_check_indices).
struct CheckArgs {
    const int32_t *page_table;
    int64_t pt_stride;
    int32_t pt_width, batch;
    const int32_t *lens;          // [batch] page-table positions each request reads
    const int32_t *out_loc;       // [n_out] or nullptr
    int32_t n_out, num_rows;
    uint32_t *counts;             // [3], zeroed by the caller's stream before the launch
};
cudaError_t launch_check_indices(const CheckArgs &a, cudaStream_t s);
// Count page-table entries of the shared prefix that differ from the first
// row's and requests shorter than the prefix (counts[0], counts[1], zeroed first).
cudaError_t launch_check_shared_prefix(const int32_t *page_table, int32_t batch, int64_t pt_stride,
                                       int32_t shared_len, const int32_t *lens, uint32_t *counts,
                                       cudaStream_t s);

int device_sm_count();

// Sets the calling thread's minisgl_last_error() message and returns `code`.
int report_error(int code, const char *msg);

// Number of bounded waits that ran out in tensor-core kernels since load
// (synchronous copy from a device counter).
cudaError_t read_kernel_timeouts(unsigned int *count);

}  // namespace minisgl
