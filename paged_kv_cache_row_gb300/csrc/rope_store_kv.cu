// rope_store_kv.cu -- rotary position embedding of q and k, fused with the
// store of k and v into the paged pool.
//
// Operation ("mini-sglang architecture deep dive", section 7.3 RoPE: a
// float32 table of [cos | sin] per position, rotary_dim = head_dim, q and k
// rotated by the angles of each token's position; mini-sglang-learn, paged
// KV pool chapter, store_kv passage: each layer then scatters the new K/V
// rows to out_loc).  For token i at position p = positions[i], every q head
// and every k head x is rotated pairwise, element j with element j + d/2:
//     y[j]       = x[j] cos_j(p) - x[j + d/2] sin_j(p)
//     y[j + d/2] = x[j + d/2] cos_j(p) + x[j] sin_j(p),      j < d/2,
// in fp32 from the bf16 inputs, rounded to bf16.  The rotated q replaces q in
// place (the attention kernels read it next); the rotated k goes straight to
// row out_loc[i] of the layer's K array and v to the same row of V.  The k
// input itself is left as it was: in the unfused engine the rotated key is
// read only by store_kv, so writing it back would be traffic for nothing.
//
// Layout of the work: a (token, head slot) unit is served by d/16 threads;
// thread t takes the 16-byte chunk t of the first half of the head and chunk
// t of the second half, i.e. the eight pairs (8t+e, d/2+8t+e).  Head slots run
// over the H_q query heads, then the H_kv key heads, then the H_kv value heads
// of a token, and consecutive threads take consecutive units, so each warp
// reads and writes whole contiguous head rows.  The cos/sin row of a token
// (d float32) is read by all of its heads and stays in L1/L2.  HBM-bound:
// 4 d (H_q + 2 H_kv + 1) + 8 bytes per token.
#include "kernels.h"
#include "ptx.cuh"

namespace minisgl {

namespace {

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float4 ld_nc_f4(const float *p) {
    uint4 u = ld_nc_v4(p);
    return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                       __uint_as_float(u.w));
}

// rotate the pairs held in the 16-byte words a (first half) and b (second half)
__device__ __forceinline__ void rotate8(uint4 &a, uint4 &b, const float (&c)[8], const float (&s)[8]) {
    uint32_t *pa = &a.x, *pb = &b.x;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float x1l = bf_lo(pa[w]), x1h = bf_hi(pa[w]);
        const float x2l = bf_lo(pb[w]), x2h = bf_hi(pb[w]);
        const int e = 2 * w;
        const float y1l = fmaf(x1l, c[e], -x2l * s[e]), y1h = fmaf(x1h, c[e + 1], -x2h * s[e + 1]);
        const float y2l = fmaf(x2l, c[e], x1l * s[e]), y2h = fmaf(x2h, c[e + 1], x1h * s[e + 1]);
        pa[w] = pack_bf16x2(y1l, y1h);
        pb[w] = pack_bf16x2(y2l, y2h);
    }
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(256) rope_store_kv_kernel(RopeStoreArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    constexpr int TPH = D / 16;  // threads per head
    constexpr int HALF = D / 2;
    const int slots = a.num_q_heads + 2 * a.num_kv_heads;
    const int64_t per_tok = (int64_t)slots * TPH;
    const int64_t total = (int64_t)a.n_tokens * per_tok;
    for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < total;
         w += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = w / per_tok;
        const int rem = (int)(w - i * per_tok);
        const int slot = rem / TPH;
        const int t = rem - slot * TPH;
        const int e0 = 8 * t;  // first element of this thread's pairs
        if (slot >= a.num_q_heads + a.num_kv_heads) {  // value head: copy into the pool
            const int h = slot - a.num_q_heads - a.num_kv_heads;
            int row = __ldg(a.out_loc + i);
            row = min(max(row, 0), a.num_rows - 1);  // out-of-range rows are a caller error
            const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(a.v) + i * a.v_tok_stride +
                                       (int64_t)h * D + e0;
            __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.v_layer) + (int64_t)row * a.row_stride +
                                 (int64_t)h * D + e0;
            st_v4(dst, ld_nc_v4(src));
            st_v4(dst + HALF, ld_nc_v4(src + HALF));
            continue;
        }
        int pos = __ldg(a.positions + i);
        pos = min(max(pos, 0), a.max_positions - 1);  // likewise a caller error
        const float *cs = a.cos_sin + (int64_t)pos * D + e0;
        float c[8], s[8];
        {
            const float4 c0 = ld_nc_f4(cs), c1 = ld_nc_f4(cs + 4);
            const float4 s0 = ld_nc_f4(cs + HALF), s1 = ld_nc_f4(cs + HALF + 4);
            c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
            c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
            s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w;
            s[4] = s1.x; s[5] = s1.y; s[6] = s1.z; s[7] = s1.w;
        }
        if (slot < a.num_q_heads) {  // query head: rotate in place
            __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(a.q) + i * a.q_tok_stride +
                               (int64_t)slot * D + e0;
            uint4 x1 = *reinterpret_cast<const uint4 *>(p);
            uint4 x2 = *reinterpret_cast<const uint4 *>(p + HALF);
            rotate8(x1, x2, c, s);
            st_v4(p, x1);
            st_v4(p + HALF, x2);
        } else {  // key head: rotate into the pool
            const int h = slot - a.num_q_heads;
            int row = __ldg(a.out_loc + i);
            row = min(max(row, 0), a.num_rows - 1);
            const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(a.k) + i * a.k_tok_stride +
                                       (int64_t)h * D + e0;
            uint4 x1 = ld_nc_v4(src), x2 = ld_nc_v4(src + HALF);
            rotate8(x1, x2, c, s);
            __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.k_layer) + (int64_t)row * a.row_stride +
                                 (int64_t)h * D + e0;
            st_v4(dst, x1);
            st_v4(dst + HALF, x2);
        }
    }
}

cudaError_t launch_rope_store_kv(const RopeStoreArgs &a, cudaStream_t s) {
    if (a.n_tokens == 0) return cudaSuccess;
    const int slots = a.num_q_heads + 2 * a.num_kv_heads;
    const int64_t total = (int64_t)a.n_tokens * slots * (a.head_dim / 16);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (a.head_dim == 128)
        return launch_pdl(rope_store_kv_kernel<128>, dim3((unsigned)blocks), dim3(256), 0, s, a);
    return launch_pdl(rope_store_kv_kernel<64>, dim3((unsigned)blocks), dim3(256), 0, s, a);
}

}  // namespace minisgl
