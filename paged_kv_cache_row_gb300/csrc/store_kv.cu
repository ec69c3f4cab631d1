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

// log2_per_tok >= 0: the chunks per token (2 * row chunks) are a power of two
// and the token / chunk split is a shift (the common case); otherwise a
// 32-bit division.  Work indices are 32-bit (the host checks the total).
__global__ void __launch_bounds__(STORE_THREADS) store_kv_kernel(StoreArgs a, int log2_per_tok) {
    pdl_wait();
    pdl_launch_dependents();
    const uint32_t chunks = (uint32_t)a.row_elems / 8;  // 16-byte chunks per row
    const uint32_t per_tok = 2u * chunks;                // K then V
    const uint32_t total = (uint32_t)a.n_tokens * per_tok;
    constexpr uint32_t SPAN = (uint32_t)STORE_U * STORE_THREADS;
    for (uint32_t base = blockIdx.x * SPAN; base < total; base += gridDim.x * SPAN) {
        uint4 val[STORE_U];
        __nv_bfloat16 *dst[STORE_U];
#pragma unroll
        for (int u = 0; u < STORE_U; ++u) {
            const uint32_t w = base + u * STORE_THREADS + threadIdx.x;
            dst[u] = nullptr;
            if (w < total) {
                const uint32_t i = log2_per_tok >= 0 ? w >> log2_per_tok : w / per_tok;
                const uint32_t rem = w - i * per_tok;
                const bool is_v = rem >= chunks;
                const uint32_t c = is_v ? rem - chunks : rem;
                int row = __ldg(a.out_loc + i);
                // out-of-range rows are a caller error; clamp so the write stays in the pool
                row = min(max(row, 0), a.num_rows - 1);
                const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(is_v ? a.v : a.k) +
                                           (int64_t)i * (is_v ? a.v_tok_stride : a.k_tok_stride) + c * 8;
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
    const int64_t per_tok = 2 * (a.row_elems / 8);
    const int64_t total = (int64_t)a.n_tokens * per_tok;
    if (total >= (int64_t(1) << 31)) return cudaErrorInvalidValue;  // the host refuses this first
    int log2_per_tok = -1;
    if ((per_tok & (per_tok - 1)) == 0)
        for (log2_per_tok = 0; (int64_t(1) << log2_per_tok) < per_tok; ++log2_per_tok) {
        }
    // one wave: as many CTAs as can be resident (8 per SM at 256 threads)
    int64_t blocks = (total + STORE_U * STORE_THREADS - 1) / (STORE_U * STORE_THREADS);
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(store_kv_kernel, dim3((unsigned)blocks), dim3(STORE_THREADS), 0, s, a, log2_per_tok);
}

}  // namespace minisgl
