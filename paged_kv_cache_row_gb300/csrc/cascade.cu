// cascade.cu -- decode attention for a batch whose requests share a cached
// prefix (the radix-cache case), reading the shared K/V once per batch.
//
// Operation: exactly minisgl_decode_attn (deep dive 5.3 PagedAttention;
// mini-sglang-learn, paged KV pool and attention-backend chapters), for a
// batch in which every request's first P page-table entries are the same
// physical rows (mini-sglang-learn, radix-cache chapter: requests that match
// a cached prefix point at the prefix's rows instead of copying them).
//
// Decomposition (softmax over a union of disjoint key ranges = log-sum-exp
// merge of the per-range results, the split-KV identity):
//   * prefix: all B decode queries against positions [0, P) of the shared
//     rows.  That is a dense multi-query block -- for KV head g, B*G query
//     rows against the same keys -- so it runs on the tensor cores in the
//     extend kernel's prefix-only mode: one pseudo-request per chunk of the
//     prefix (its page-table row starts at the chunk's first column, so the
//     row stride is the chunk length), all of them reading q rows 0..B-1 and
//     writing fp32 partial outputs and LSEs to their own rows.  Chunks are
//     sized so the launch has about two work items per SM.
//   * suffix: each request's own positions [P, n_r) with the split-KV decode
//     kernels (page table shifted by P columns, context n_r - P), which also
//     return each row's LSE.
//   * merge: per (request, query head), the prefix chunks and the suffix are
//     combined by their LSEs and written as bf16.
// A setup kernel writes the pseudo-requests' lengths and offsets into the
// caller's workspace, so the call allocates nothing and never synchronises.
#include "kernels.h"
#include "ptx.cuh"

namespace minisgl {

namespace {

// pseudo-request metadata of the prefix launch and the suffix lengths
__global__ void cascade_setup_kernel(CascadeArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int B = a.batch, S = a.chunks;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < B + S + 1; i += gridDim.x * blockDim.x) {
        if (i < S) {  // prefix chunk i
            a.meta.pre_cached[i] = min(a.chunk_len, a.shared_len - i * a.chunk_len);
            a.meta.pre_extend[i] = B;
            a.meta.pre_qoff[i] = 0;
            a.meta.pre_ooff[i] = i * B;
        } else if (i < S + B) {  // suffix of request r
            const int r = i - S;
            a.meta.suf_seq[r] = max(__ldg(a.seq_lens + r) - a.shared_len, 0);
        } else {
            a.meta.pre_qoff[S] = B;
        }
    }
}

// one warp per (request, query head): merge the S prefix partials (fp32) and
// the suffix result (bf16, weight 0 when its LSE is -inf: empty suffix)
template <int D>
__global__ void __launch_bounds__(256) cascade_merge_kernel(CascadeArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    constexpr int PER = D / 32;  // channels per lane
    const int lane = threadIdx.x & 31;
    const int64_t nvec = (int64_t)a.batch * a.num_q_heads;
    for (int64_t v = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; v < nvec;
         v += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        // lane p < S holds prefix chunk p's LSE
        const float lp = lane < a.chunks ? a.pre_lse[(int64_t)lane * nvec + v] : -INFINITY;
        const float ls = a.suf_lse[v];
        float top = fmaxf(lp, ls);
#pragma unroll
        for (int o = 16; o; o >>= 1) top = fmaxf(top, __shfl_xor_sync(0xffffffffu, top, o));
        const float wp = lane < a.chunks ? __expf(lp - top) : 0.f;
        const float ws = ls == -INFINITY ? 0.f : __expf(ls - top);
        float total = wp;
#pragma unroll
        for (int o = 16; o; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
        total += ws;
        float acc[PER];
        {
            const __nv_bfloat16 *so = static_cast<const __nv_bfloat16 *>(a.suf_out) + v * D + lane * PER;
#pragma unroll
            for (int c = 0; c < PER; ++c) acc[c] = ws * __bfloat162float(so[c]);
        }
        for (int p = 0; p < a.chunks; ++p) {
            const float w = __shfl_sync(0xffffffffu, wp, p);
            const float *o = a.pre_o + ((int64_t)p * nvec + v) * D + lane * PER;
#pragma unroll
            for (int c = 0; c < PER; c += 4) {
                const float4 x = *reinterpret_cast<const float4 *>(o + c);
                acc[c] += w * x.x;
                acc[c + 1] += w * x.y;
                acc[c + 2] += w * x.z;
                acc[c + 3] += w * x.w;
            }
        }
        const float inv = 1.f / total;
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) + v * D + lane * PER;
#pragma unroll
        for (int c = 0; c < PER; c += 2)
            *reinterpret_cast<uint32_t *>(dst + c) = pack_bf16x2(acc[c] * inv, acc[c + 1] * inv);
    }
}

}  // namespace

cudaError_t launch_cascade(const CascadeArgs &c, const ExtendArgs &base, cudaStream_t s) {
    if (c.batch == 0) return cudaSuccess;
    cudaError_t e = launch_pdl(cascade_setup_kernel, dim3(1), dim3(256), 0, s, c);
    if (e != cudaSuccess) return e;
    // prefix: one pseudo-request per chunk, rows of the shared prefix
    ExtendArgs p = base;
    p.page_table = c.page_table;
    p.pt_stride = c.chunk_len;
    p.pt_width = c.chunk_len;
    p.batch = c.chunks;
    p.total_q_tokens = c.chunks * c.batch;
    p.cached_lens = c.meta.pre_cached;
    p.extend_lens = c.meta.pre_extend;
    p.q_offsets = c.meta.pre_qoff;
    p.out_offsets = c.meta.pre_ooff;
    p.prefix_only = 1;
    p.out_f32 = c.pre_o;
    p.lse_out = c.pre_lse;
    if ((e = launch_extend(p, s)) != cudaSuccess) return e;
    // suffix: split-KV decode over each request's own positions, with LSEs
    if ((e = launch_decode(c.suffix, s)) != cudaSuccess) return e;
    const int64_t warps = (int64_t)c.batch * c.num_q_heads;
    int64_t blocks = (warps * 32 + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(cascade_merge_kernel<128>, dim3((unsigned)blocks), dim3(256), 0, s, c);
}

}  // namespace minisgl
