// decode.cu -- split-KV GQA decode attention over the paged pool, and the
// log-sum-exp merge of its partial results.
//
// What it computes (mini-sglang-learn, paged KV pool chapter: page_table rows
// hold raw physical rows; attention-backend chapter: decode is memory bound
// and parallelises over the KV length, the FlashDecoding idea; deep dive
// section 5.3, PagedAttention): for request r and query head h of KV group g,
//     out[r,h] = sum_j softmax_j(sm_scale <q[r,h], K[pt[r,j], g]>) V[pt[r,j], g],  j < seq_len[r].
//
// Design (GB300):
//   * Work = the concatenation, over requests r and KV heads g, of "streams"
//     (r, g) of 16-token tiles.  The total tile count is cut into equal
//     contiguous segments, one per warp of a persistent grid sized to the
//     SMs, so every warp moves the same number of bytes whatever the length
//     mix (a long request is split over several warps, short ones share a
//     warp).  Each CTA derives the same schedule from seq_lens on its own
//     (a prefix sum in shared memory), so no planning pass or host sync is
//     needed.
//   * Each warp runs its own STAGES-deep cp.async ring: a tile is the K and V
//     rows of 16 tokens for one KV head (plus the group's queries when the
//     tile opens a stream), gathered through page_table with 16-byte copies
//     into XOR-swizzled shared memory.  Page-table entries are fetched one
//     tile ahead of the copies that need them.
//   * The group's query heads (G <= 8 padded to 8 rows, else 16) form the M
//     side of warp-level bf16 tensor-core MMAs: S = Q K^T (m16n8k16) and
//     O += P V; the online softmax runs in fp32 on the accumulator
//     fragments, in base 2.
//   * A warp whose segment covers a whole stream writes the bf16 output; a
//     stream cut across segments leaves normalised fp32 partials and their
//     natural-log LSE in the workspace, and decode_merge_kernel combines them.
#include <cfloat>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace minisgl {

namespace {

constexpr int TILE = 16;  // tokens per warp tile
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

template <int D, int MROWS>
struct Cfg {
    static constexpr int RB = D * 2;             // bytes of one head row
    static constexpr int CPR = RB / 16;          // 16-byte chunks per row
    static constexpr int KV_BYTES = TILE * RB;   // one K (or V) tile
    static constexpr int Q_BYTES = MROWS * RB;   // the group's queries
    static constexpr int STAGE_BYTES = 2 * KV_BYTES + Q_BYTES;
    static constexpr int NT = D / 8;             // n8 tiles along head_dim
    static constexpr int KS = D / 16;            // k16 steps along head_dim
};

struct Cursor {
    int r, g, j, nt, n;  // request, kv head, tile in stream, tiles in stream, tokens
};

__device__ __forceinline__ int clamp_len(int n, int w) { return min(max(n, 0), w); }

// Swizzled byte offset of 16-byte chunk cc of row t inside a tile.
__device__ __forceinline__ uint32_t swz(int t, int cc, int rb) {
    return (uint32_t)(t * rb + ((cc ^ (t & 7)) << 4));
}

}  // namespace

template <int D, int MROWS, int WARPS, int STAGES>
__global__ void __launch_bounds__(WARPS * 32)
    decode_partial_kernel(const DecodeArgs a, const float scale_log2, const int prefix_bytes) {
    using C = Cfg<D, MROWS>;
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ int s_maxtiles;
    int32_t *s_prefix = reinterpret_cast<int32_t *>(smem);

    const int B = a.batch, Hkv = a.num_kv_heads, Hq = a.num_q_heads, W = a.pt_width;
    const int G = Hq / Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- schedule: prefix over requests of (tiles per stream) * Hkv -------
    if (warp == 0) {
        int carry = 0, mx = 0;
        if (lane == 0) s_prefix[0] = 0;
        for (int base = 0; base < B; base += 32) {
            const int r = base + lane;
            int nt = 0;
            if (r < B) nt = (clamp_len(__ldg(a.seq_lens + r), W) + TILE - 1) / TILE;
            mx = max(mx, nt);
            int v = nt * Hkv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (r < B) s_prefix[r + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) s_maxtiles = mx;
    }
    __syncthreads();
    const int total = s_prefix[B];
    const int nwarps = gridDim.x * WARPS;
    int P = a.split_tokens > 0 ? (a.split_tokens + TILE - 1) / TILE : (total + nwarps - 1) / nwarps;
    P = max(P, 1);
    // at most max_splits partials per stream: ceil(nt / P) + 1 <= max_splits
    P = max(P, (s_maxtiles + a.max_splits - 2) / (a.max_splits - 1));

    const __nv_bfloat16 *Kl = static_cast<const __nv_bfloat16 *>(a.k_layer);
    const __nv_bfloat16 *Vl = static_cast<const __nv_bfloat16 *>(a.v_layer);
    const __nv_bfloat16 *Q = static_cast<const __nv_bfloat16 *>(a.q);
    const uint32_t ring = smem_u32(smem + prefix_bytes) + warp * STAGES * C::STAGE_BYTES;

    auto locate = [&](Cursor &c, int t) {
        int lo = 0, hi = B;  // largest r with prefix[r] <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_prefix[mid] <= t) lo = mid; else hi = mid;
        }
        c.r = lo;
        c.n = clamp_len(__ldg(a.seq_lens + lo), W);
        c.nt = (c.n + TILE - 1) / TILE;
        const int off = t - s_prefix[lo];
        c.g = off / c.nt;
        c.j = off - c.g * c.nt;
    };
    auto advance = [&](Cursor &c) {  // only called when a next tile exists
        if (++c.j == c.nt) {
            c.j = 0;
            if (++c.g == Hkv) {
                c.g = 0;
                do { ++c.r; } while (s_prefix[c.r + 1] == s_prefix[c.r]);
                c.n = clamp_len(__ldg(a.seq_lens + c.r), W);
                c.nt = (c.n + TILE - 1) / TILE;
            }
        }
    };
    // lane < 16: physical row of token 16*j + lane of the cursor's request, or -1 past its end
    auto load_rows = [&](const Cursor &c) -> int {
        const int tok = c.j * TILE + lane;
        if (lane >= TILE || tok >= c.n) return -1;
        const int row = __ldg(a.page_table + (int64_t)c.r * a.pt_stride + tok);
        return min(max(row, 0), a.num_rows - 1);
    };
    auto issue = [&](int stage, const Cursor &c, int rows, bool with_q) {
        const uint32_t st = ring + stage * C::STAGE_BYTES;
        const int64_t head = (int64_t)c.g * D;
#pragma unroll
        for (int i = 0; i < TILE * C::CPR / 32; ++i) {
            const int ch = lane + 32 * i;
            const int tt = ch / C::CPR, cc = ch % C::CPR;
            const int row = __shfl_sync(0xffffffffu, rows, tt);
            const uint32_t off = swz(tt, cc, C::RB);
            const int64_t e = (int64_t)max(row, 0) * a.row_stride + head + cc * 8;
            const int bytes = row >= 0 ? 16 : 0;
            cp_async_16(st + off, Kl + e, bytes);
            cp_async_16(st + C::KV_BYTES + off, Vl + e, bytes);
        }
        if (with_q) {
#pragma unroll
            for (int i = 0; i < MROWS * C::CPR / 32; ++i) {
                const int ch = lane + 32 * i;
                const int qi = ch / C::CPR, cc = ch % C::CPR;
                const bool live = qi < G;
                const __nv_bfloat16 *src =
                    live ? Q + ((int64_t)c.r * Hq + c.g * G + qi) * D + cc * 8 : Q;
                cp_async_16(st + 2 * C::KV_BYTES + swz(qi, cc, C::RB), src, live ? 16 : 0);
            }
        }
    };

    for (int64_t seg = (int64_t)blockIdx.x * WARPS + warp; seg * P < total; seg += nwarps) {
        const int t0 = (int)(seg * P);
        const int t1 = min(t0 + P, total);

        Cursor pc, cc;
        locate(pc, t0);
        cc = pc;
        // prologue: first STAGES-1 tiles
#pragma unroll
        for (int s = 0; s < STAGES - 1; ++s) {
            if (t0 + s < t1) {
                const int rows = load_rows(pc);
                issue(s, pc, rows, s == 0 || pc.j == 0);
                if (t0 + s + 1 < t1) advance(pc);
            }
            cp_async_commit();
        }
        int rows_next = (t0 + STAGES - 1 < t1) ? load_rows(pc) : -1;

        // consumer state
        int cur_r = -1, cur_g = 0, cur_nt = 0, cur_start = 0, first_j = 0, last_j = 0;
        float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
        float o[C::NT][4];
        uint32_t qa[C::KS][4];

        auto flush = [&]() {
            float lr0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
            lr0 += __shfl_xor_sync(0xffffffffu, lr0, 2);
            float lr1 = 0.f;
            if (MROWS == 16) {
                lr1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
                lr1 += __shfl_xor_sync(0xffffffffu, lr1, 2);
            }
            const bool last = last_j == cur_nt - 1;
            const bool whole = first_j == 0 && last;
            const int hl = lane >> 2, c2 = 2 * (lane & 3);
            const int s = whole ? 0 : (int)(seg - cur_start / P);
#pragma unroll
            for (int half = 0; half < (MROWS == 16 ? 2 : 1); ++half) {
                const int row = hl + 8 * half;
                if (row >= G) continue;
                const float lr = half ? lr1 : lr0, mr = half ? m1 : m0;
                const float inv = 1.f / lr;
                const int64_t hh = (int64_t)cur_r * Hq + cur_g * G + row;
                if (whole) {
                    __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) + hh * D + c2;
#pragma unroll
                    for (int dt = 0; dt < C::NT; ++dt)
                        *reinterpret_cast<uint32_t *>(dst + 8 * dt) =
                            pack_bf16x2(o[dt][2 * half] * inv, o[dt][2 * half + 1] * inv);
                } else {
                    float *dst = a.ws_o + (hh * a.max_splits + s) * D + c2;
#pragma unroll
                    for (int dt = 0; dt < C::NT; ++dt)
                        *reinterpret_cast<float2 *>(dst + 8 * dt) =
                            make_float2(o[dt][2 * half] * inv, o[dt][2 * half + 1] * inv);
                    if ((lane & 3) == 0) a.ws_lse[hh * a.max_splits + s] = (mr + __log2f(lr)) * LN2;
                }
            }
            if (last && lane == 0) a.split_count[(int64_t)cur_r * Hkv + cur_g] = s + 1;
        };

        for (int t = t0; t < t1; ++t) {
            const int tp = t + STAGES - 1;
            if (tp < t1) {
                issue((tp - t0) % STAGES, pc, rows_next, pc.j == 0);
                if (tp + 1 < t1) {
                    advance(pc);
                    rows_next = load_rows(pc);
                }
            }
            cp_async_commit();
            cp_async_wait<STAGES - 1>();
            __syncwarp();

            const uint32_t st = ring + ((t - t0) % STAGES) * C::STAGE_BYTES;
            if (cc.r != cur_r || cc.g != cur_g) {
                if (cur_r >= 0) flush();
                cur_r = cc.r;
                cur_g = cc.g;
                cur_nt = cc.nt;
                cur_start = s_prefix[cc.r] + cc.g * cc.nt;
                first_j = cc.j;
                m0 = m1 = -INFINITY;
                l0 = l1 = 0.f;
#pragma unroll
                for (int dt = 0; dt < C::NT; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
                // query fragments (A operand, rows = heads of the group)
                const uint32_t qs = st + 2 * C::KV_BYTES;
                if (MROWS == 8) {
#pragma unroll
                    for (int ks = 0; ks < C::KS; ks += 2) {
                        const int row = lane & 7, ch = 2 * ks + (lane >> 3);
                        ldsm_x4(qs + swz(row, ch, C::RB), qa[ks][0], qa[ks][2], qa[ks + 1][0],
                                qa[ks + 1][2]);
                        qa[ks][1] = qa[ks][3] = qa[ks + 1][1] = qa[ks + 1][3] = 0u;
                    }
                } else {
#pragma unroll
                    for (int ks = 0; ks < C::KS; ++ks) {
                        const int row = (lane & 7) + ((lane >> 3) & 1) * 8, ch = 2 * ks + (lane >> 4);
                        ldsm_x4(qs + swz(row, ch, C::RB), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
                    }
                }
            }

            // S = Q K^T for 16 tokens: two n8 tiles
            float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int ks = 0; ks < C::KS; ++ks) {
                const int tok = ((lane >> 4) << 3) + (lane & 7), ch = 2 * ks + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(st + swz(tok, ch, C::RB), b0, b1, b2, b3);
                mma_bf16_16816(s[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                mma_bf16_16816(s[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
            }
            // online softmax (base 2), rows hl and hl+8
            const int tok0 = cc.j * TILE + 2 * (lane & 3);
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const bool ok = tok0 + 8 * nt + e < cc.n;
                    s[nt][e] = ok ? s[nt][e] * scale_log2 : -INFINITY;
                    s[nt][2 + e] = ok ? s[nt][2 + e] * scale_log2 : -INFINITY;
                    mx0 = fmaxf(mx0, s[nt][e]);
                    mx1 = fmaxf(mx1, s[nt][2 + e]);
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            const float mn0 = fmaxf(m0, mx0);
            const float al0 = ex2(m0 - mn0);
            m0 = mn0;
            float ps = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    s[nt][e] = ex2(s[nt][e] - mn0);
                    ps += s[nt][e];
                }
            l0 = l0 * al0 + ps;
            float al1 = 1.f;
            if (MROWS == 16) {
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                const float mn1 = fmaxf(m1, mx1);
                al1 = ex2(m1 - mn1);
                m1 = mn1;
                float ps1 = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        s[nt][2 + e] = ex2(s[nt][2 + e] - mn1);
                        ps1 += s[nt][2 + e];
                    }
                l1 = l1 * al1 + ps1;
            }
            // P as the A operand (rows = heads, k = the 16 tokens)
            const uint32_t pa0 = pack_bf16x2(s[0][0], s[0][1]);
            const uint32_t pa2 = pack_bf16x2(s[1][0], s[1][1]);
            const uint32_t pa1 = MROWS == 16 ? pack_bf16x2(s[0][2], s[0][3]) : 0u;
            const uint32_t pa3 = MROWS == 16 ? pack_bf16x2(s[1][2], s[1][3]) : 0u;
            // O = O * alpha + P V
#pragma unroll
            for (int dt = 0; dt < C::NT; dt += 2) {
                o[dt][0] *= al0; o[dt][1] *= al0; o[dt + 1][0] *= al0; o[dt + 1][1] *= al0;
                if (MROWS == 16) {
                    o[dt][2] *= al1; o[dt][3] *= al1; o[dt + 1][2] *= al1; o[dt + 1][3] *= al1;
                }
                const int tok = ((lane >> 3) & 1) * 8 + (lane & 7), ch = dt + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(st + C::KV_BYTES + swz(tok, ch, C::RB), b0, b1, b2, b3);
                mma_bf16_16816(o[dt], pa0, pa1, pa2, pa3, b0, b1);
                mma_bf16_16816(o[dt + 1], pa0, pa1, pa2, pa3, b2, b3);
            }
            last_j = cc.j;
            if (t + 1 < t1) advance(cc);
            __syncwarp();
        }
        if (cur_r >= 0) flush();
        cp_async_wait<0>();
        __syncwarp();
    }
}

// One CTA per (request, KV head); thread c owns channel c of every head of
// the group.  Streams that one warp finished are left alone (their bf16
// output is final); empty requests get zeros.
template <int D>
__global__ void __launch_bounds__(D) decode_merge_kernel(const DecodeArgs a) {
    const int Hkv = a.num_kv_heads, Hq = a.num_q_heads, G = Hq / Hkv;
    const int r = blockIdx.x / Hkv, g = blockIdx.x - r * Hkv;
    const int c = threadIdx.x;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out);
    const int n = min(max(__ldg(a.seq_lens + r), 0), a.pt_width);
    if (n == 0) {
        for (int i = 0; i < G; ++i)
            out[((int64_t)r * Hq + g * G + i) * D + c] = __float2bfloat16_rn(0.f);
        return;
    }
    const int S = min(a.split_count[(int64_t)r * Hkv + g], a.max_splits);
    if (S <= 1) return;
    for (int i = 0; i < G; ++i) {
        const int64_t base = ((int64_t)r * Hq + g * G + i) * a.max_splits;
        float M = -INFINITY;
        for (int s = 0; s < S; ++s) M = fmaxf(M, a.ws_lse[base + s]);
        float tot = 0.f, acc = 0.f;
        for (int s = 0; s < S; ++s) {
            const float w = __expf(a.ws_lse[base + s] - M);
            tot += w;
            acc += w * a.ws_o[(base + s) * D + c];
        }
        out[((int64_t)r * Hq + g * G + i) * D + c] = __float2bfloat16_rn(acc / tot);
    }
}

namespace {

struct LaunchCache {
    std::mutex mu;
    struct Entry { const void *fn; int dev; size_t smem; int blocks; };
    Entry e[64];
    int n = 0;
};
LaunchCache g_cache;

template <typename K>
int blocks_per_sm(K kernel, int threads, size_t smem) {
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(g_cache.mu);
    for (int i = 0; i < g_cache.n; ++i)
        if (g_cache.e[i].fn == (const void *)kernel && g_cache.e[i].dev == dev &&
            g_cache.e[i].smem == smem)
            return g_cache.e[i].blocks;
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, threads, smem) != cudaSuccess)
        nb = 0;
    if (g_cache.n < 64) g_cache.e[g_cache.n++] = {(const void *)kernel, dev, smem, nb};
    return nb;
}

template <int D, int MROWS>
cudaError_t launch_cfg(const DecodeArgs &a, cudaStream_t s) {
    constexpr int WARPS = 4, STAGES = 4;
    using C = Cfg<D, MROWS>;
    const int prefix_bytes = (((a.batch + 1) * 4) + 1023) / 1024 * 1024;
    const size_t smem = (size_t)prefix_bytes + (size_t)WARPS * STAGES * C::STAGE_BYTES;
    auto kern = decode_partial_kernel<D, MROWS, WARPS, STAGES>;
    const int nb = blocks_per_sm(kern, WARPS * 32, smem);
    if (nb <= 0) return cudaErrorInvalidConfiguration;
    // never more warps than tiles could exist
    const int64_t max_tiles = (int64_t)a.batch * a.num_kv_heads * ((a.pt_width + TILE - 1) / TILE);
    int64_t grid = (int64_t)device_sm_count() * nb;
    const int64_t need = (max_tiles + WARPS - 1) / WARPS;
    if (grid > need) grid = need;
    if (grid < 1) grid = 1;
    kern<<<(unsigned)grid, WARPS * 32, smem, s>>>(a, a.sm_scale * LOG2E, prefix_bytes);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_merge_kernel<D><<<a.batch * a.num_kv_heads, D, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s) {
    if (a.batch == 0) return cudaSuccess;
    const int G = a.num_q_heads / a.num_kv_heads;
    if (a.head_dim == 128) return G <= 8 ? launch_cfg<128, 8>(a, s) : launch_cfg<128, 16>(a, s);
    return G <= 8 ? launch_cfg<64, 8>(a, s) : launch_cfg<64, 16>(a, s);
}

}  // namespace minisgl
