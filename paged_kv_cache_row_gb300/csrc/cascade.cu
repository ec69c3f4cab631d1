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
//     extend kernel's prefix-chunk mode: chunk c covers shared positions
//     [c*chunk_len, (c+1)*chunk_len) of the first page-table row, every chunk
//     reads q rows 0..B-1 and writes fp32 partial outputs and LSEs to its own
//     rows.  The chunk geometry is arithmetic, so no metadata is written.
//   * suffix: each request's own positions [P, n_r) with the split-KV decode
//     partial kernel (page table shifted by P columns, context n_r - P),
//     which leaves fp32 partials and LSEs for every stream, split or not.
//   * merge: per (request, query head), the prefix chunks and the suffix
//     splits are combined by their LSEs in fp32 and written as bf16.
// The two parts are independent.  When the prefix launch leaves enough SMs
// free, the suffix runs on a library-owned second stream, forked from and
// joined back to the caller's stream with events (capturable in a CUDA
// graph), on those free SMs only, so both parts run at the same time.
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace minisgl {

namespace {

// one warp per (request, query head): merge the prefix chunks' fp32 partials
// (lane c holds chunk c's LSE) and the suffix's split partials (lane s holds
// split s's LSE; none when the request has no private positions).  Loads come
// in two batches: first the context length, the split count and everything
// of the prefix (LSEs and up to PF rows), which do not depend on the split
// count; then the suffix LSEs and rows (at most SMAX).
template <int D>
__global__ void __launch_bounds__(256) cascade_merge_kernel(CascadeArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    constexpr int PER = D / 32;  // channels per lane: 4 (d 128) or 2 (d 64)
    static_assert(PER == 4 || PER == 2, "head_dim 64 or 128");
    constexpr int PF = 8;        // prefix rows loaded in the first round
    constexpr int SMAX = 16;     // suffix splits (the cascade call uses 16)
    const int lane = threadIdx.x & 31;
    const DecodeArgs &sd = a.suffix;
    const int G = a.num_q_heads / sd.num_kv_heads;
    const int64_t nvec = (int64_t)a.batch * a.num_q_heads;
    auto load_row = [&](const float *o, float (&x)[PER]) {
        if constexpr (PER == 4) {
            const float4 t = *reinterpret_cast<const float4 *>(o);
            x[0] = t.x, x[1] = t.y, x[2] = t.z, x[3] = t.w;
        } else {
            const float2 t = *reinterpret_cast<const float2 *>(o);
            x[0] = t.x, x[1] = t.y;
        }
    };
    for (int64_t v = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; v < nvec;
         v += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        const int r = (int)(v / a.num_q_heads), h = (int)(v - (int64_t)r * a.num_q_heads);
        // first loads: nothing here depends on the split count
        const int seq = __ldg(a.seq_lens + r);
        const int cnt = sd.split_count[(int64_t)r * sd.num_kv_heads + h / G];  // stale if no suffix: unused then
        const float lp = lane < a.chunks ? a.pre_lse[(int64_t)lane * nvec + v] : -INFINITY;
        float xp[PF][PER];
#pragma unroll
        for (int k = 0; k < PF; ++k) {
            if (k < a.chunks) load_row(a.pre_o + ((int64_t)k * nvec + v) * D + lane * PER, xp[k]);
            else
#pragma unroll
                for (int c = 0; c < PER; ++c) xp[k][c] = 0.f;
        }
        // second loads: the suffix splits
        const int n_suf = min(max(seq - a.shared_len, 0), sd.pt_width);
        const int S = n_suf > 0 ? min(min(cnt, sd.max_splits), SMAX) : 0;
        const int64_t sbase = v * sd.max_splits;
        const float ls = lane < S ? sd.ws_lse[sbase + lane] : -INFINITY;
        float xs[SMAX][PER];
#pragma unroll
        for (int k = 0; k < SMAX; ++k) {
            if (k < S) load_row(sd.ws_o + (sbase + k) * D + lane * PER, xs[k]);
            else
#pragma unroll
                for (int c = 0; c < PER; ++c) xs[k][c] = 0.f;
        }
        float top = fmaxf(lp, ls);
#pragma unroll
        for (int o = 16; o; o >>= 1) top = fmaxf(top, __shfl_xor_sync(0xffffffffu, top, o));
        const float wp = lane < a.chunks ? __expf(lp - top) : 0.f;
        const float ws = lane < S ? __expf(ls - top) : 0.f;
        float total = wp + ws;
#pragma unroll
        for (int o = 16; o; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
        float acc[PER];
#pragma unroll
        for (int c = 0; c < PER; ++c) acc[c] = 0.f;
#pragma unroll
        for (int k = 0; k < PF; ++k) {
            const float w = __shfl_sync(0xffffffffu, wp, k);  // 0 past the chunks
#pragma unroll
            for (int c = 0; c < PER; ++c) acc[c] += w * xp[k][c];
        }
        for (int k = PF; k < a.chunks; ++k) {  // more than PF chunks: one row at a time
            float x[PER];
            load_row(a.pre_o + ((int64_t)k * nvec + v) * D + lane * PER, x);
            const float w = __shfl_sync(0xffffffffu, wp, k);
#pragma unroll
            for (int c = 0; c < PER; ++c) acc[c] += w * x[c];
        }
#pragma unroll
        for (int k = 0; k < SMAX; ++k) {
            const float w = __shfl_sync(0xffffffffu, ws, k);  // 0 past S
#pragma unroll
            for (int c = 0; c < PER; ++c) acc[c] += w * xs[k][c];
        }
        const float inv = 1.f / total;
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) + v * D + lane * PER;
#pragma unroll
        for (int c = 0; c < PER; c += 2)
            *reinterpret_cast<uint32_t *>(dst + c) = pack_bf16x2(acc[c] * inv, acc[c + 1] * inv);
    }
}

// A second stream per device and the two events that fork work onto it and
// join it back, created on first use.  The mutex is held while a call
// enqueues its fork, its side-stream launch and its join, so calls from
// several host threads do not interleave their uses of the events.
struct Side {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;
Side g_side[64];

cudaError_t side_for_current_device(Side **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    Side &sd = g_side[dev];
    if (!sd.stream) {  // all three, or none (a failed creation is retried by the next call)
        Side n;
        if ((e = cudaStreamCreateWithFlags(&n.stream, cudaStreamNonBlocking)) == cudaSuccess &&
            (e = cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming)) == cudaSuccess &&
            (e = cudaEventCreateWithFlags(&n.join, cudaEventDisableTiming)) == cudaSuccess) {
            sd = n;
        } else {
            if (n.fork) cudaEventDestroy(n.fork);
            if (n.stream) cudaStreamDestroy(n.stream);
            return e;
        }
    }
    *out = &sd;
    return cudaSuccess;
}

// SMs the suffix needs at least before it is worth running beside the prefix
constexpr int MIN_FREE_SMS = 24;

}  // namespace

cudaError_t launch_cascade(const CascadeArgs &c, const ExtendArgs &prefix, cudaStream_t s) {
    if (c.batch == 0) return cudaSuccess;
    const int sms = device_sm_count();
    const int free_sms = sms - extend_grid(prefix);
    const int64_t warps = (int64_t)c.batch * c.num_q_heads;
    int64_t blocks = (warps * 32 + 255) / 256;
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    auto merge = [&]() {
        return c.head_dim == 64
                   ? launch_pdl(cascade_merge_kernel<64>, dim3((unsigned)blocks), dim3(256), 0, s, c)
                   : launch_pdl(cascade_merge_kernel<128>, dim3((unsigned)blocks), dim3(256), 0, s, c);
    };
    cudaError_t e;
    if (free_sms < MIN_FREE_SMS) {  // one after the other on the caller's stream
        if ((e = launch_extend(prefix, s)) != cudaSuccess) return e;
        if ((e = launch_decode(c.suffix, s)) != cudaSuccess) return e;
        return merge();
    }
    std::lock_guard<std::mutex> lk(g_side_mu);
    Side *side = nullptr;
    if ((e = side_for_current_device(&side)) != cudaSuccess) return e;
    // the prefix goes first, so its CTAs take their SMs before the suffix's
    // are placed; the suffix is limited to the SMs left over
    if ((e = cudaEventRecord(side->fork, s)) != cudaSuccess) return e;
    if ((e = launch_extend(prefix, s)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(side->stream, side->fork, 0)) != cudaSuccess) return e;
    DecodeArgs suf = c.suffix;
    suf.max_sms = free_sms;
    if ((e = launch_decode(suf, side->stream)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(side->join, side->stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(s, side->join, 0)) != cudaSuccess) return e;
    return merge();
}

}  // namespace minisgl
