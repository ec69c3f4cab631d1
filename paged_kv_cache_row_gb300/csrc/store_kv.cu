// store_kv.cu -- scatter new K/V token rows into the paged pool.
//
// Operation (mini-sglang-learn, paged KV pool chapter, store_kv passage;
// deep dive section 6.2 MHAKVCache): for every new token i, its K row and its
// V row (num_kv_heads * head_dim bf16 each) are copied to physical row
// out_loc[i] of the layer's K and V arrays.
//
// The reference store kernel gives one warp to each token row.  Here the unit
// is a 16-byte vector: consecutive threads take consecutive 16-byte chunks of
// the same row, so every warp moves 512 contiguous bytes per instruction on
// both the read and the write side, whatever the row length.  A CTA covers
// U * 256 consecutive chunks per pass: each thread loads its U chunks (U
// independent 16-byte loads in flight) before storing them.  The kernel is a
// pure HBM copy: 2 * row_bytes read + 2 * row_bytes written + 4 index bytes
// per token.
#include "kernels.h"
#include "ptx.cuh"

namespace minisgl {

namespace {
constexpr int STORE_THREADS = 256;
constexpr int STORE_U = 4;  // chunks per thread per pass
}  // namespace

__global__ void __launch_bounds__(STORE_THREADS) store_kv_kernel(StoreArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int chunks = a.row_elems / 8;                  // 16-byte chunks per row
    const int64_t per_tok = 2LL * chunks;                // K then V
    const int64_t total = (int64_t)a.n_tokens * per_tok;
    constexpr int64_t SPAN = (int64_t)STORE_U * STORE_THREADS;
    for (int64_t base = (int64_t)blockIdx.x * SPAN; base < total; base += (int64_t)gridDim.x * SPAN) {
        uint4 val[STORE_U];
        __nv_bfloat16 *dst[STORE_U];
#pragma unroll
        for (int u = 0; u < STORE_U; ++u) {
            const int64_t w = base + u * STORE_THREADS + threadIdx.x;
            dst[u] = nullptr;
            if (w < total) {
                const int64_t i = w / per_tok;
                const int rem = (int)(w - i * per_tok);
                const int is_v = rem >= chunks;
                const int c = is_v ? rem - chunks : rem;
                int row = __ldg(a.out_loc + i);
                // out-of-range rows are a caller error; clamp so the write stays in the pool
                row = min(max(row, 0), a.num_rows - 1);
                const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(is_v ? a.v : a.k) +
                                           i * (is_v ? a.v_tok_stride : a.k_tok_stride) + c * 8;
                dst[u] = static_cast<__nv_bfloat16 *>(is_v ? a.v_layer : a.k_layer) +
                         (int64_t)row * a.row_stride + c * 8;
                val[u] = ld_nc_v4(src);
            }
        }
#pragma unroll
        for (int u = 0; u < STORE_U; ++u)
            if (dst[u]) st_v4(dst[u], val[u]);
    }
}

cudaError_t launch_store_kv(const StoreArgs &a, cudaStream_t s) {
    if (a.n_tokens == 0) return cudaSuccess;
    const int64_t total = (int64_t)a.n_tokens * 2 * (a.row_elems / 8);
    int64_t blocks = (total + STORE_U * STORE_THREADS - 1) / (STORE_U * STORE_THREADS);
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (blocks > cap) blocks = cap;
    return launch_pdl(store_kv_kernel, dim3((unsigned)blocks), dim3(STORE_THREADS), 0, s, a);
}

}  // namespace minisgl
