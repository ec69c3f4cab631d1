// extend.cu -- causal attention for chunked-prefill (extend) tokens over the
// paged pool, on the Blackwell tensor cores (tcgen05, fp32 accumulators in
// tensor memory).
//
// What it computes (mini-sglang-learn: request-state passage, extend_len =
// device_len - cached_len; chunked-prefill chapter; attention-backend chapter:
// prefill is compute bound and wants large tensor-core tiles; SGLang source
// reading guide: ForwardBatch extend_prefix_lens / extend_seq_lens): new token
// t of request r sits at position C_r + t and attends to logical tokens
// 0 .. C_r + t of its page_table row:
//     out[q_off[r]+t, h] = sum_{j <= C_r+t} softmax_j(sm_scale <q, K[pt[r,j], g]>) V[pt[r,j], g].
//
// Design (GB300, one CTA per SM, persistent):
//   * Work item = (request, KV head g, block of TQ = 128/G new tokens).  The
//     128 MMA rows are the (token, head) pairs of the block: the G query
//     heads that share KV head g ride in the same tile, so each gathered K/V
//     tile feeds G heads.
//   * Producer warps 4-7 gather 128-token K and V tiles through page_table
//     with 16-byte cp.async into the 128-byte-swizzled layout the tensor
//     core reads (K as a K-major B operand, V as an MN-major B operand), two
//     stages deep; completion is tracked by mbarriers
//     (cp.async.mbarrier.arrive).
//   * Warp 8 (one lane) issues tcgen05.mma: S = Q K^T (M=N=128, K=16 steps)
//     into one of two S buffers in TMEM, then O += P V into a TMEM O buffer,
//     and signals completions with tcgen05.commit.
//   * Softmax warps 0-3: thread i owns TMEM lane (= MMA row) i.  It reads its
//     S row, applies the causal limit C + t, keeps a running max m and sum l
//     (base 2), writes P = 2^(s - m) as bf16 into shared memory for the PV
//     MMA, and rescales its O row in TMEM only when the max has grown by
//     more than 2^8 (the final O / l is unchanged by when the rescale
//     happens).  Epilogue: O / l -> bf16 -> global.
//   * Every mbarrier wait is bounded in time; a wait that runs out sets a
//     flag, the kernel finishes without further waiting (its output is then
//     garbage) and the device counter minisgl_timeouts is increased.
#include <mutex>

#include "kernels.h"
#include "tcgen05.cuh"

namespace minisgl {

__device__ unsigned int g_kernel_timeouts = 0;

namespace {

constexpr int D = 128;
constexpr int ROWS = 128;                 // MMA M and KV tile length
constexpr int TILE_BYTES = ROWS * D * 2;  // 32 KB: 128 rows of 256 bytes
constexpr int HALF = TILE_BYTES / 2;      // one 64-column swizzle region
constexpr int OFF_Q = 0;
constexpr int OFF_P = TILE_BYTES;
constexpr int OFF_KV = 2 * TILE_BYTES;    // stage s: K at +2s*TILE, V at +(2s+1)*TILE
constexpr int STAGES = 2;
constexpr int OFF_BAR = OFF_KV + STAGES * 2 * TILE_BYTES;  // 192 KB
constexpr int OFF_TMEM_SLOT = OFF_BAR + 96;
constexpr int OFF_PREFIX = OFF_BAR + 128;
constexpr int THREADS = 288;              // 4 softmax + 4 producer + 1 MMA warp
constexpr int MMA_WARP = 8;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O = 256;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_LOG2 = 8.f;
constexpr long long WAIT_LIMIT = 4000000000LL;  // SM cycles (about 2 s)

// byte offset of 16-byte chunk cc (0..15) of row `row` in a 128 x 256 B tile
// stored as two 128-byte-swizzled 64-column regions
__device__ __forceinline__ uint32_t sw128(int row, int cc) {
    return (uint32_t)((cc >> 3) * HALF + (row >> 3) * 1024 + (row & 7) * 128 +
                      (((cc & 7) ^ (row & 7)) << 4));
}

// Bounded mbarrier wait shared by all roles: once one wait has run out, the
// CTA stops waiting altogether so every thread reaches the end quickly.
__device__ __forceinline__ void guarded_wait(uint32_t b, uint32_t parity, int *abort_flag) {
    if (*((volatile int *)abort_flag)) return;
    if (!mbar_wait(b, parity, WAIT_LIMIT)) {
        *((volatile int *)abort_flag) = 1;
        atomicAdd(&g_kernel_timeouts, 1u);
    }
}

__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}

}  // namespace

__global__ void __launch_bounds__(THREADS, 1)
    extend_kernel(const ExtendArgs a, const float scale_log2, const int log2g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ int s_abort;
    const uint32_t sb = smem_u32(base);
    const uint32_t sQ = sb + OFF_Q, sP = sb + OFF_P, sKV = sb + OFF_KV;
    const uint32_t bar = sb + OFF_BAR;
    auto kv_full = [&](int s) { return bar + 8 * s; };
    auto kv_empty = [&](int s) { return bar + 16 + 8 * s; };
    auto s_full = [&](int b) { return bar + 32 + 8 * b; };
    const uint32_t p_full = bar + 48, pv_done = bar + 56, fin = bar + 64;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + OFF_TMEM_SLOT);
    int32_t *s_prefix = reinterpret_cast<int32_t *>(base + OFF_PREFIX);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = a.batch, Hkv = a.num_kv_heads, Hq = a.num_q_heads, W = a.pt_width;
    const int G = 1 << log2g;
    const int TQ = ROWS >> log2g;  // new tokens per work item

    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(kv_full(s), 128);
            mbar_init(kv_empty(s), 1);
        }
        mbar_init(s_full(0), 1);
        mbar_init(s_full(1), 1);
        mbar_init(p_full, 128);
        mbar_init(pv_done, 1);
        mbar_init(fin, 1);
        fence_mbar_init();
        s_abort = 0;
    }
    if (warp == MMA_WARP) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    // items per request: ceil(E / TQ) blocks times Hkv heads, prefix in shared memory
    if (warp == 4) {
        int carry = 0;
        if (lane == 0) s_prefix[0] = 0;
        for (int b0 = 0; b0 < B; b0 += 32) {
            const int r = b0 + lane;
            int v = 0;
            if (r < B) {
                const int c = min(max(__ldg(a.cached_lens + r), 0), W);
                const int e = min(max(__ldg(a.extend_lens + r), 0), W - c);
                v = ((e + TQ - 1) / TQ) * Hkv;
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (r < B) s_prefix[r + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int total_items = s_prefix[B];

#define wait(b, parity) guarded_wait((b), (parity), &s_abort)

    const __nv_bfloat16 *Kl = static_cast<const __nv_bfloat16 *>(a.k_layer);
    const __nv_bfloat16 *Vl = static_cast<const __nv_bfloat16 *>(a.v_layer);
    const __nv_bfloat16 *Q = static_cast<const __nv_bfloat16 *>(a.q);
    const uint32_t idesc_qk = idesc_bf16_f32(ROWS, ROWS, false);
    const uint32_t idesc_pv = idesc_bf16_f32(ROWS, D, true);

    uint32_t kv_iter = 0;  // KV tiles this CTA has gone through (all roles count alike)
    for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
        int lo = 0, hi = B;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_prefix[mid] <= item) lo = mid; else hi = mid;
        }
        const int r = lo;
        const int nqb = (s_prefix[r + 1] - s_prefix[r]) / Hkv;
        const int off = item - s_prefix[r];
        const int g = off / nqb, qb = off - g * nqb;
        const int C = min(max(__ldg(a.cached_lens + r), 0), W);
        const int E = min(max(__ldg(a.extend_lens + r), 0), W - C);
        const int qoff = __ldg(a.q_offsets + r);
        const int t_first = qb * TQ;
        const int t_last = min(t_first + TQ, E) - 1;
        const int n_vis = C + t_last + 1;  // KV positions this block can see
        const int nkv = (n_vis + ROWS - 1) / ROWS;

        if (warp >= 4 && warp < 8) {
            // ---------------- producer: Q once, then K/V tiles ----------------
            // Thread pt copies 16-byte chunk cc of rows tb*16 .. tb*16+15 of each
            // 128-row tile (16 threads cover one 256-byte row).  The page-table
            // entries of the next tile are fetched while this tile's copies go out.
            const int pt = threadIdx.x - 128;
            const int cc = pt & 15, tb = pt >> 4;
            const int32_t *ptab = a.page_table + (int64_t)r * a.pt_stride;
            auto fetch_rows = [&](int j, int (&rows)[16]) {
                const int p0 = j * ROWS + tb * 16;
                if (p0 + 16 <= n_vis && ((reinterpret_cast<uintptr_t>(ptab + p0) & 15) == 0)) {
                    const int4 *src = reinterpret_cast<const int4 *>(ptab + p0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int4 v = __ldg(src + q);
                        rows[4 * q + 0] = v.x;
                        rows[4 * q + 1] = v.y;
                        rows[4 * q + 2] = v.z;
                        rows[4 * q + 3] = v.w;
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 16; ++k) rows[k] = p0 + k < n_vis ? __ldg(ptab + p0 + k) : -1;
                }
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    rows[k] = rows[k] < 0 ? -1 : min(rows[k], a.num_rows - 1);
            };
            int rows_cur[16], rows_nxt[16];
            fetch_rows(0, rows_nxt);
            for (int j = 0; j < nkv; ++j) {
#pragma unroll
                for (int k = 0; k < 16; ++k) rows_cur[k] = rows_nxt[k];
                if (j + 1 < nkv) fetch_rows(j + 1, rows_nxt);
                const uint32_t it = kv_iter + j, st = it & 1;
                if (it >= STAGES) wait(kv_empty(st), ((it >> 1) - 1) & 1);
                if (j == 0) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int i = tb * 16 + k;
                        const int t = t_first + (i >> log2g);
                        const bool live = t <= t_last;
                        const __nv_bfloat16 *src =
                            live ? Q + ((int64_t)(qoff + t) * Hq + g * G + (i & (G - 1))) * D + cc * 8
                                 : Q;
                        cp_async_16(sQ + sw128(i, cc), src, live ? 16 : 0);
                    }
                }
                const uint32_t sK = sKV + st * 2 * TILE_BYTES, sV = sK + TILE_BYTES;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int tok = tb * 16 + k;
                    const int row = rows_cur[k];
                    const int64_t e = (int64_t)max(row, 0) * a.row_stride + (int64_t)g * D + cc * 8;
                    const int bytes = row >= 0 ? 16 : 0;
                    const uint32_t o = sw128(tok, cc);
                    cp_async_16(sK + o, Kl + e, bytes);
                    cp_async_16(sV + o, Vl + e, bytes);
                }
                cp_async_mbar_arrive_noinc(kv_full(st));
            }
            cp_async_wait<0>();
        } else if (warp == MMA_WARP) {
            // ---------------- MMA issuer ----------------
            if (lane == 0) {
                // S(j) is issued one tile ahead of PV(j-1), so the S MMA of the next
                // tile runs while the softmax warps work on the current one.
                for (int j = 0; j <= nkv; ++j) {
                    if (j < nkv) {
                        const uint32_t it = kv_iter + j, st = it & 1;
                        wait(kv_full(st), (it >> 1) & 1);
                        fence_proxy_async_smem();
                        tc_fence_after();
                        const uint32_t sK = sKV + st * 2 * TILE_BYTES;
                        const uint32_t dS = tmem + ((it & 1) ? COL_S1 : COL_S0);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint64_t ad = smem_desc_sw128(sQ + (kk >> 2) * HALF + (kk & 3) * 32, 16, 1024);
                            const uint64_t bd = smem_desc_sw128(sK + (kk >> 2) * HALF + (kk & 3) * 32, 16, 1024);
                            tc_mma_bf16(dS, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
                        }
                        tc_commit(s_full(it & 1));
                    }
                    if (j > 0) {
                        const int jj = j - 1;
                        const uint32_t itp = kv_iter + jj, st = itp & 1;
                        wait(p_full, itp & 1);
                        tc_fence_after();
                        const uint32_t sV = sKV + st * 2 * TILE_BYTES + TILE_BYTES;
#pragma unroll
                        for (int kk = 0; kk < ROWS / 16; ++kk) {
                            const uint64_t ad = smem_desc_sw128(sP + (kk >> 2) * HALF + (kk & 3) * 32, 16, 1024);
                            const uint64_t bd = smem_desc_sw128(sV + kk * 2048, HALF, 1024);
                            tc_mma_bf16(tmem + COL_O, ad, bd, idesc_pv, (jj > 0 || kk > 0) ? 1u : 0u);
                        }
                        tc_commit(pv_done);
                        tc_commit(kv_empty(st));
                    }
                }
            }
            __syncwarp();
        } else {
            // ---------------- softmax / epilogue: thread i owns row i ----------------
            const int i = threadIdx.x;
            const int t = min(t_first + (i >> log2g), t_last);
            const bool live = t_first + (i >> log2g) <= t_last;
            const int lim = C + t;  // last visible position
            const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < nkv; ++j) {
                const uint32_t it = kv_iter + j;
                wait(s_full(it & 1), (it >> 1) & 1);
                tc_fence_after();
                const uint32_t scol = lane_base + ((it & 1) ? COL_S1 : COL_S0);
                const int pos0 = j * ROWS;
                // pass 1: row max of the scaled, masked scores (32 columns at a time)
                float mx = -INFINITY;
#pragma unroll 1
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t sr[32];
                    tmem_ld32(scol + 32 * q4, sr);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (pos0 + 32 * q4 + c <= lim) mx = fmaxf(mx, __uint_as_float(sr[c]) * scale_log2);
                }
                const float m_new = fmaxf(m, mx);
                if (j > 0) {
                    wait(pv_done, (it - 1) & 1);  // PV(j-1) done: P buffer free, O settled
                    tc_fence_after();
                    if (__any_sync(0xffffffffu, m_new > m + RESCALE_LOG2)) {
                        const float alpha = ex2(m - m_new);
                        l *= alpha;
                        m = m_new;
#pragma unroll 1
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint32_t o[32];
                            tmem_ld32(lane_base + COL_O + 32 * q4, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                            tmem_st32(lane_base + COL_O + 32 * q4, o);
                        }
                        tmem_wait_st();
                    }
                } else {
                    m = m_new;
                }
                // pass 2: P = 2^(s - m) as bf16 into row i of the P tile
#pragma unroll 1
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t sr[32];
                    tmem_ld32(scol + 32 * q4, sr);
                    tmem_wait_ld();
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = 8 * c8 + 2 * e;
                            const int p = pos0 + 32 * q4 + c;
                            const float p0 = p <= lim ? ex2(__uint_as_float(sr[c]) * scale_log2 - m) : 0.f;
                            const float p1 = p + 1 <= lim ? ex2(__uint_as_float(sr[c + 1]) * scale_log2 - m) : 0.f;
                            l += p0 + p1;
                            w[e] = pack_bf16x2(p0, p1);
                        }
                        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(sP + sw128(i, 4 * q4 + c8)),
                                     "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                                     : "memory");
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(p_full);
            }
            // epilogue: O / l -> bf16
            wait(pv_done, (kv_iter + nkv - 1) & 1);
            tc_fence_after();
            const float inv = 1.f / l;
            __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) +
                                 ((int64_t)(qoff + t) * Hq + g * G + (i & (G - 1))) * D;
#pragma unroll 1
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t o[32];
                tmem_ld32(lane_base + COL_O + 32 * q4, o);
                tmem_wait_ld();
                if (live) {
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(o[c + 0]) * inv, __uint_as_float(o[c + 1]) * inv);
                        v.y = pack_bf16x2(__uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
                        v.z = pack_bf16x2(__uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv);
                        v.w = pack_bf16x2(__uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv);
                        *reinterpret_cast<uint4 *>(dst + 32 * q4 + c) = v;
                    }
                }
            }
            tc_fence_before();
        }
        kv_iter += nkv;
        named_bar_sync(1, THREADS);  // item done: MMAs finished, O read, Q free
        tc_fence_after();
    }

#undef wait
    // drain anything still in flight before TMEM is released
    if (warp == MMA_WARP) {
        if (lane == 0) {
            tc_commit(fin);
            if (!mbar_wait(fin, 0, WAIT_LIMIT)) atomicAdd(&g_kernel_timeouts, 1u);
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == MMA_WARP) tmem_dealloc(tmem, TMEM_COLS);
}

cudaError_t launch_extend(const ExtendArgs &a, cudaStream_t s) {
    if (a.batch == 0 || a.total_q_tokens == 0) return cudaSuccess;
    const int G = a.num_q_heads / a.num_kv_heads;
    int log2g = 0;
    while ((1 << log2g) < G) ++log2g;
    const int TQ = ROWS >> log2g;
    const size_t smem = (size_t)OFF_PREFIX + (size_t)(a.batch + 1) * 4 + 1024;
    static std::mutex mu;
    static bool configured[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lk(mu);
        if (dev >= 0 && dev < 64 && !configured[dev]) {
            cudaError_t e = cudaFuncSetAttribute(extend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 OFF_PREFIX + 4097 * 4 + 1024);
            if (e != cudaSuccess) return e;
            configured[dev] = true;
        }
    }
    // upper bound on work items: every request can add one partial block
    const int64_t items = ((int64_t)a.total_q_tokens / TQ + a.batch) * a.num_kv_heads;
    int64_t grid = device_sm_count();
    if (grid > items) grid = items;
    if (grid < 1) grid = 1;
    return launch_pdl(extend_kernel, dim3((unsigned)grid), dim3(THREADS), smem, s, a,
                      a.sm_scale * LOG2E, log2g);
}

cudaError_t read_kernel_timeouts(unsigned int *count) {
    return cudaMemcpyFromSymbol(count, g_kernel_timeouts, sizeof(unsigned int));
}

}  // namespace minisgl
