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
//   * For the shared-prefix (cascade) call: a length offset (a request's row
//     starts past the shared positions), fp32 partials for whole streams too
//     with no merge launch (the cascade merge combines them with the prefix
//     part), and a grid limited to the SMs the prefix part leaves free.
#include <cfloat>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace minisgl {

namespace {

constexpr int TILE = 16;  // tokens per warp tile
constexpr int MAX_WARPS = 12;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

template <int D>
struct Cfg {
    static constexpr int RB = D * 2;            // bytes of one head row
    static constexpr int CPR = RB / 16;         // 16-byte chunks per row
    static constexpr int KV_BYTES = TILE * RB;  // one K (or V) tile
    static constexpr int KS = D / 16;           // k16 steps along head_dim (QK^T)
    static constexpr int MT = D / 16;           // m16 tiles along head_dim (PV)
};

struct Cursor {
    int r, g, j, nt, n;  // request, kv head, tile in stream, tiles in stream, tokens
};

__device__ __forceinline__ int clamp_len(int n, int w) { return min(max(n, 0), w); }

// Swizzled byte offset of 16-byte chunk cc of row t inside a K or V tile.
__device__ __forceinline__ uint32_t swz(int t, int cc, int rb) {
    return (uint32_t)(t * rb + ((cc ^ (t & 7)) << 4));
}

// Transpose an 8x8 b16 matrix held in the mma fragment layout.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

}  // namespace

// NG: n8 tiles of query heads (1 when the group has <= 8 heads, else 2).
// The MMAs put the 16 tokens of a tile on M and the group's heads on N:
//   S^T[tok, h] = K[tok, :] . Q[h, :]      (A = K tile, B = Q)
//   O^T[c, h]  += V^T[c, tok] P^T[tok, h]  (A = V tile transposed, B = P^T)
// so a group of 8 heads fills the MMA with no padding rows.
template <int D, int NG, int STAGES>
__global__ void __launch_bounds__(MAX_WARPS * 32, 1)
    decode_partial_kernel(const DecodeArgs a, const float scale_log2, const int prefix_bytes,
                          const int stage_bytes) {
    using C = Cfg<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    int32_t *s_prefix = reinterpret_cast<int32_t *>(smem);  // [B + 1], then the longest stream
    int32_t &s_maxtiles = s_prefix[a.batch + 1];

    const int B = a.batch, Hkv = a.num_kv_heads, Hq = a.num_q_heads, W = a.pt_width;
    const int G = Hq / Hkv;
    const int WARPS = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_launch_dependents();

    // ---- schedule: prefix over requests of (tiles per stream) * Hkv -------
    if (warp == 0) {
        int carry = 0, mx = 0;
        if (lane == 0) s_prefix[0] = 0;
        for (int base = 0; base < B; base += 32) {
            const int r = base + lane;
            int nt = 0;
            if (r < B) nt = (clamp_len(__ldg(a.seq_lens + r) - a.len_offset, W) + TILE - 1) / TILE;
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
    const uint32_t ring = smem_u32(smem + prefix_bytes) + warp * STAGES * stage_bytes;

    auto locate = [&](Cursor &c, int t) {
        int lo = 0, hi = B;  // largest r with prefix[r] <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_prefix[mid] <= t) lo = mid; else hi = mid;
        }
        c.r = lo;
        c.n = clamp_len(__ldg(a.seq_lens + lo) - a.len_offset, W);
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
                c.n = clamp_len(__ldg(a.seq_lens + c.r) - a.len_offset, W);
                c.nt = (c.n + TILE - 1) / TILE;
            }
        }
    };
    // lane < 16: physical row of token 16*j + lane of the cursor's request, or -1 past its
    // end; with the fused store, -2 for a position whose row is the request's out_loc row
    // (its K/V are read from this step's new rows, which this kernel is storing there)
    auto load_rows = [&](const Cursor &c) -> int {
        const int tok = c.j * TILE + lane;
        if (lane >= TILE || tok >= c.n) return -1;
        const int row = min(max(__ldg(a.page_table + (int64_t)c.r * a.pt_stride + tok), 0), a.num_rows - 1);
        if (a.out_loc && row == min(max(__ldg(a.out_loc + c.r), 0), a.num_rows - 1)) return -2;
        return row;
    };
    // fused store_kv: this lane's 16-byte chunk of a new K/V head slice, loaded
    // when the stream's last tile is issued and written one tile later, so the
    // load's latency hides behind the tile being computed
    static_assert(2 * C::CPR <= 32, "one chunk of the new K and V head slice per lane");
    uint4 st_val = make_uint4(0u, 0u, 0u, 0u);
    __nv_bfloat16 *st_dst = nullptr;
    auto store_pending = [&]() {
        if (st_dst) st_v4(st_dst, st_val);
        st_dst = nullptr;
    };
    // K and V rows of one tile (plus the group's queries when the tile opens a stream)
    auto issue = [&](int stage, const Cursor &c, int rows, bool with_q) {
        const uint32_t st = ring + stage * stage_bytes;
        const int64_t head = (int64_t)c.g * D;
#pragma unroll
        for (int i = 0; i < TILE * C::CPR / 32; ++i) {
            const int ch = lane + 32 * i;
            const int tt = ch / C::CPR, cc = ch % C::CPR;
            const int row = __shfl_sync(0xffffffffu, rows, tt);
            const uint32_t off = swz(tt, cc, C::RB);
            const int64_t e = (int64_t)max(row, 0) * a.row_stride + head + cc * 8;
            const int bytes = row != -1 ? 16 : 0;
            const __nv_bfloat16 *ks = Kl + e, *vs = Vl + e;
            if (row == -2) {
                ks = static_cast<const __nv_bfloat16 *>(a.k_new) + (int64_t)c.r * a.new_k_stride + head + cc * 8;
                vs = static_cast<const __nv_bfloat16 *>(a.v_new) + (int64_t)c.r * a.new_v_stride + head + cc * 8;
            }
            cp_async_16(st + off, ks, bytes);
            cp_async_16(st + C::KV_BYTES + off, vs, bytes);
        }
        if (a.out_loc && c.j == c.nt - 1) {
            // fused store_kv: the warp that reads a stream's last tile writes the
            // request's new K and V head slice to its out_loc row (lane < CPR: K
            // chunk, else V chunk)
            store_pending();
            const int row = min(max(__ldg(a.out_loc + c.r), 0), a.num_rows - 1);
            if (lane < 2 * C::CPR) {
                const bool isv = lane >= C::CPR;
                const int cc = isv ? lane - C::CPR : lane;
                const __nv_bfloat16 *src =
                    static_cast<const __nv_bfloat16 *>(isv ? a.v_new : a.k_new) +
                    (int64_t)c.r * (isv ? a.new_v_stride : a.new_k_stride) + head + cc * 8;
                st_val = ld_nc_v4(src);
                st_dst = const_cast<__nv_bfloat16 *>(isv ? Vl : Kl) + (int64_t)row * a.row_stride +
                         head + cc * 8;
            }
        }
        if (with_q) {
            const __nv_bfloat16 *src = Q + ((int64_t)c.r * Hq + c.g * G) * D;
            for (int ch = lane; ch < G * C::CPR; ch += 32)
                cp_async_16(st + 2 * C::KV_BYTES + ch * 16, src + ch * 8, 16);
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
        // page-table rows two tiles ahead of the copies that need them
        Cursor pl = pc;
        int rows_a = -1, rows_b = -1;
        if (t0 + STAGES - 1 < t1) {
            rows_a = load_rows(pl);
            if (t0 + STAGES < t1) {
                advance(pl);
                rows_b = load_rows(pl);
            }
        }

        // consumer state: per head column e of n-tile n, running max m and lane-partial sum l
        int cur_r = -1, cur_g = 0, cur_nt = 0, cur_start = 0, first_j = 0, last_j = 0;
        float m[NG][2], l[NG][2];
        float o[C::MT][NG][4];
        uint32_t qb[NG][C::KS][2];

        auto flush = [&]() {
            const bool last = last_j == cur_nt - 1;
            const bool whole = first_j == 0 && last;
            const int s = whole ? 0 : (int)(seg - cur_start / P);
            const int dr = lane >> 2;
#pragma unroll
            for (int n = 0; n < NG; ++n)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float lt = l[n][e];
                    lt += __shfl_xor_sync(0xffffffffu, lt, 4);
                    lt += __shfl_xor_sync(0xffffffffu, lt, 8);
                    lt += __shfl_xor_sync(0xffffffffu, lt, 16);
                    const int h = n * 8 + 2 * (lane & 3) + e;
                    if (h >= G) continue;
                    const float inv = 1.f / lt;
                    const int64_t hh = (int64_t)cur_r * Hq + cur_g * G + h;
                    if (whole && !a.partials_only) {
                        if (a.lse_out && dr == 0) a.lse_out[hh] = (m[n][e] + __log2f(lt)) * LN2;
                        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) + hh * D + dr;
#pragma unroll
                        for (int mt = 0; mt < C::MT; ++mt) {
                            dst[16 * mt] = __float2bfloat16_rn(o[mt][n][e] * inv);
                            dst[16 * mt + 8] = __float2bfloat16_rn(o[mt][n][2 + e] * inv);
                        }
                    } else {
                        float *dst = a.ws_o + (hh * a.max_splits + s) * D + dr;
#pragma unroll
                        for (int mt = 0; mt < C::MT; ++mt) {
                            dst[16 * mt] = o[mt][n][e] * inv;
                            dst[16 * mt + 8] = o[mt][n][2 + e] * inv;
                        }
                        if (dr == 0) a.ws_lse[hh * a.max_splits + s] = (m[n][e] + __log2f(lt)) * LN2;
                    }
                }
            if (last && lane == 0) a.split_count[(int64_t)cur_r * Hkv + cur_g] = s + 1;
        };

        for (int t = t0; t < t1; ++t) {
            const int tp = t + STAGES - 1;
            if (tp < t1) {
                issue((tp - t0) % STAGES, pc, rows_a, pc.j == 0);
                if (tp + 1 < t1) {
                    advance(pc);
                    rows_a = rows_b;
                    if (tp + 2 < t1) {
                        advance(pl);
                        rows_b = load_rows(pl);
                    }
                }
            }
            cp_async_commit();
            cp_async_wait<STAGES - 1>();
            __syncwarp();

            const uint32_t st = ring + ((t - t0) % STAGES) * stage_bytes;
            if (cc.r != cur_r || cc.g != cur_g) {
                if (cur_r >= 0) flush();
                cur_r = cc.r;
                cur_g = cc.g;
                cur_nt = cc.nt;
                cur_start = s_prefix[cc.r] + cc.g * cc.nt;
                first_j = cc.j;
#pragma unroll
                for (int n = 0; n < NG; ++n) {
                    m[n][0] = m[n][1] = -INFINITY;
                    l[n][0] = l[n][1] = 0.f;
                }
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
                    for (int n = 0; n < NG; ++n) o[mt][n][0] = o[mt][n][1] = o[mt][n][2] = o[mt][n][3] = 0.f;
                // Q as the B operand: b0 = Q[h][16ks + 2(l%4) + {0,1}], b1 = the same + 8
                const uint32_t qs = st + 2 * C::KV_BYTES;
#pragma unroll
                for (int n = 0; n < NG; ++n) {
                    const int h = n * 8 + (lane >> 2);
#pragma unroll
                    for (int ks = 0; ks < C::KS; ++ks) {
                        uint32_t b0 = 0u, b1 = 0u;
                        if (h < G) {
                            const uint32_t ad = qs + h * C::RB + (16 * ks + 2 * (lane & 3)) * 2;
                            asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(b0) : "r"(ad));
                            asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(b1) : "r"(ad + 16));
                        }
                        qb[n][ks][0] = b0;
                        qb[n][ks][1] = b1;
                    }
                }
            }

            // S^T = K Q^T for the tile's 16 tokens; two accumulator chains per n-tile
            float sa[NG][2][4];
#pragma unroll
            for (int n = 0; n < NG; ++n)
#pragma unroll
                for (int c = 0; c < 2; ++c) sa[n][c][0] = sa[n][c][1] = sa[n][c][2] = sa[n][c][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < C::KS; ++ks) {
                const int tok = (lane & 7) + ((lane >> 3) & 1) * 8, ch = 2 * ks + (lane >> 4);
                uint32_t a0, a1, a2, a3;
                ldsm_x4(st + swz(tok, ch, C::RB), a0, a1, a2, a3);
#pragma unroll
                for (int n = 0; n < NG; ++n)
                    mma_bf16_16816(sa[n][ks & 1], a0, a1, a2, a3, qb[n][ks][0], qb[n][ks][1]);
            }
            // online softmax per head column, base 2; this lane holds tokens
            // dr and dr + 8 of the tile for heads 2(l%4) and 2(l%4)+1
            const int tokA = cc.j * TILE + (lane >> 2);
            const bool okA = tokA < cc.n, okB = tokA + 8 < cc.n;
            uint32_t pb[NG][2];
#pragma unroll
            for (int n = 0; n < NG; ++n) {
                float p[4];
                float al[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float x0 = okA ? (sa[n][0][e] + sa[n][1][e]) * scale_log2 : -INFINITY;
                    const float x1 = okB ? (sa[n][0][2 + e] + sa[n][1][2 + e]) * scale_log2 : -INFINITY;
                    float mx = fmaxf(x0, x1);
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    const float mn = fmaxf(m[n][e], mx);
                    al[e] = ex2(m[n][e] - mn);
                    m[n][e] = mn;
                    p[e] = ex2(x0 - mn);
                    p[2 + e] = ex2(x1 - mn);
                    l[n][e] = l[n][e] * al[e] + p[e] + p[2 + e];
                }
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
                    o[mt][n][0] *= al[0];
                    o[mt][n][1] *= al[1];
                    o[mt][n][2] *= al[0];
                    o[mt][n][3] *= al[1];
                }
                // P^T as the B operand: transpose the two 8x8 token-by-head blocks
                pb[n][0] = movmatrix_t(pack_bf16x2(p[0], p[1]));
                pb[n][1] = movmatrix_t(pack_bf16x2(p[2], p[3]));
            }
            // O^T += V^T P^T
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
                const int tok = (lane & 7) + (lane >> 4) * 8, ch = 2 * mt + ((lane >> 3) & 1);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(st + C::KV_BYTES + swz(tok, ch, C::RB), a0, a1, a2, a3);
#pragma unroll
                for (int n = 0; n < NG; ++n) mma_bf16_16816(o[mt][n], a0, a1, a2, a3, pb[n][0], pb[n][1]);
            }
            last_j = cc.j;
            if (t + 1 < t1) advance(cc);
            store_pending();
            __syncwarp();
        }
        store_pending();
        if (cur_r >= 0) flush();
        cp_async_wait<0>();
        __syncwarp();
    }
}

// One warp per (request, query head).  Streams that one warp of the partial
// kernel finished (split count 1) already hold their final bf16 output and are
// skipped; empty requests get zeros.  Lane s holds the weight of split s (32 at
// a time); every lane owns D/32 consecutive channels.
template <int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeArgs a) {
    constexpr int CPL = D / 32;  // channels per lane
    constexpr int PRE = 8;       // partial rows loaded before the weights are known
    const int Hkv = a.num_kv_heads, Hq = a.num_q_heads, G = Hq / Hkv;
    const int wid = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    pdl_wait();
    pdl_launch_dependents();
    if (wid >= a.batch * Hq) return;
    const int r = wid / Hq, h = wid - r * Hq, g = h / G;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out) + (int64_t)wid * D + lane * CPL;
    // dependent rounds of loads: the context length, the split count (written
    // by the partial kernel only for non-empty requests, so read after the
    // empty check), then the first 32 LSEs together with the first PRE
    // partial rows
    const int n = min(max(__ldg(a.seq_lens + r) - a.len_offset, 0), a.pt_width);
    if (n == 0) {
#pragma unroll
        for (int c = 0; c < CPL; ++c) out[c] = __float2bfloat16_rn(0.f);
        if (a.lse_out && lane == 0) a.lse_out[wid] = -INFINITY;
        return;
    }
    const int cnt = a.split_count[(int64_t)r * Hkv + g];
    const int S = min(cnt, a.max_splits);
    if (S <= 1) return;
    const int64_t base = (int64_t)wid * a.max_splits;
    const float *orow = a.ws_o + base * D + lane * CPL;  // split k at orow + k * D
    const float l0 = lane < S ? a.ws_lse[base + lane] : -INFINITY;
    float2 pre[PRE][CPL / 2];
#pragma unroll
    for (int k = 0; k < PRE; ++k)
#pragma unroll
        for (int c = 0; c < CPL / 2; ++c)
            pre[k][c] = k < S ? *reinterpret_cast<const float2 *>(orow + k * D + 2 * c) : make_float2(0.f, 0.f);
    float M = l0;
    for (int s0 = 32; s0 < S; s0 += 32)
        if (s0 + lane < S) M = fmaxf(M, a.ws_lse[base + s0 + lane]);
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float acc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
    const float w0 = lane < S ? __expf(l0 - M) : 0.f;
    float tot = w0;
#pragma unroll
    for (int k = 0; k < PRE; ++k) {
        const float wk = __shfl_sync(0xffffffffu, w0, k);  // 0 for k >= S
#pragma unroll
        for (int c = 0; c < CPL / 2; ++c) {
            acc[2 * c] += wk * pre[k][c].x;
            acc[2 * c + 1] += wk * pre[k][c].y;
        }
    }
    for (int s0 = 0; s0 < S; s0 += 32) {
        float w = w0;
        if (s0 > 0) {
            w = s0 + lane < S ? __expf(a.ws_lse[base + s0 + lane] - M) : 0.f;
            tot += w;
        }
        const int ns = min(32, S - s0);
        for (int k = s0 > 0 ? 0 : PRE; k < ns; ++k) {
            const float wk = __shfl_sync(0xffffffffu, w, k);
            const float *src = orow + (int64_t)(s0 + k) * D;
#pragma unroll
            for (int c = 0; c < CPL; c += 2) {
                const float2 v = *reinterpret_cast<const float2 *>(src + c);
                acc[c] += wk * v.x;
                acc[c + 1] += wk * v.y;
            }
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if (a.lse_out && lane == 0) a.lse_out[wid] = M + __logf(tot);
    const float inv = 1.f / tot;
#pragma unroll
    for (int c = 0; c < CPL; c += 2)
        *reinterpret_cast<uint32_t *>(out + c) = pack_bf16x2(acc[c] * inv, acc[c + 1] * inv);
}

namespace {

struct SmemInfo {
    int optin;     // dynamic + static shared memory one CTA may use
    int per_sm;    // shared memory of one SM
    int reserved;  // shared memory the system reserves per CTA
};

SmemInfo smem_info() {
    static std::mutex mu;
    static SmemInfo cache[64];
    static bool have[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    if (dev >= 0 && dev < 64 && have[dev]) return cache[dev];
    SmemInfo si{48 * 1024, 48 * 1024, 0};
    cudaDeviceGetAttribute(&si.optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaDeviceGetAttribute(&si.per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&si.reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (dev >= 0 && dev < 64) {
        cache[dev] = si;
        have[dev] = true;
    }
    return si;
}

struct LaunchCache {
    std::mutex mu;
    struct Entry { const void *fn; int dev; size_t smem; int threads; int blocks; };
    Entry e[64];
    int n = 0;
    struct Attr { const void *fn; int dev; };
    Attr a[64];
    int na = 0;
};
LaunchCache g_cache;

// CTAs per SM for `kernel` at this block size and dynamic shared memory.  The
// kernel's dynamic shared-memory limit is raised to the device maximum once
// per device, so launches with any smaller size stay valid.
template <typename K>
int blocks_per_sm(K kernel, int threads, size_t smem) {
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(g_cache.mu);
    for (int i = 0; i < g_cache.n; ++i)
        if (g_cache.e[i].fn == (const void *)kernel && g_cache.e[i].dev == dev &&
            g_cache.e[i].smem == smem && g_cache.e[i].threads == threads)
            return g_cache.e[i].blocks;
    bool attr = false;
    for (int i = 0; i < g_cache.na; ++i)
        if (g_cache.a[i].fn == (const void *)kernel && g_cache.a[i].dev == dev) attr = true;
    if (!attr) {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        const int dyn_max = smem_info().optin - (int)fa.sharedSizeBytes;
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max) !=
            cudaSuccess) {
            cudaGetLastError();  // do not leave the failure for the next caller to find
            return 0;
        }
        if (g_cache.na < 64) g_cache.a[g_cache.na++] = {(const void *)kernel, dev};
    }
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, threads, smem) != cudaSuccess) {
        cudaGetLastError();
        nb = 0;
    }
    if (g_cache.n < 64) g_cache.e[g_cache.n++] = {(const void *)kernel, dev, smem, threads, nb};
    return nb;
}

template <int D, int NG, int STAGES>
cudaError_t launch_cfg(const DecodeArgs &a, cudaStream_t s) {
    using C = Cfg<D>;
    const int G = a.num_q_heads / a.num_kv_heads;
    const int prefix_bytes = (((a.batch + 2) * 4) + 1023) / 1024 * 1024;
    const int stage_bytes = ((2 * C::KV_BYTES + G * C::RB) + 127) / 128 * 128;
    // As many warps per SM as shared memory allows (more warps hide more
    // latency), as two CTAs of at most CTA_WARPS warps when they fit.
    constexpr int CTA_WARPS = 6;
    const SmemInfo si = smem_info();
    const int per_warp = STAGES * stage_bytes;
    const int fixed = prefix_bytes + si.reserved;
    int warps = (si.per_sm - 2 * fixed) / per_warp / 2;
    if (warps < 1) warps = (si.per_sm - fixed) / per_warp;  // one CTA per SM
    if (warps > CTA_WARPS) warps = CTA_WARPS;
    while (warps > 0 && prefix_bytes + warps * per_warp > si.optin) --warps;
    if (warps < 1) return cudaErrorInvalidConfiguration;
    const size_t smem = (size_t)prefix_bytes + (size_t)warps * per_warp;
    auto kern = decode_partial_kernel<D, NG, STAGES>;
    const int nb = blocks_per_sm(kern, warps * 32, smem);
    if (nb <= 0) return cudaErrorInvalidConfiguration;
    // never more warps than tiles could exist
    const int64_t max_tiles = (int64_t)a.batch * a.num_kv_heads * ((a.pt_width + TILE - 1) / TILE);
    int64_t grid = (int64_t)device_sm_count() * nb;
    const int64_t need = (max_tiles + warps - 1) / warps;
    if (grid > need) grid = need;
    if (a.max_sms > 0 && grid > (int64_t)a.max_sms * nb) grid = (int64_t)a.max_sms * nb;
    if (grid < 1) grid = 1;
    cudaError_t e = launch_pdl(kern, dim3((unsigned)grid), dim3(warps * 32), smem, s, a,
                               a.sm_scale * LOG2E, prefix_bytes, stage_bytes);
    if (e != cudaSuccess || a.partials_only) return e;
    return launch_pdl(decode_merge_kernel<D>, dim3((a.batch * a.num_q_heads + 3) / 4), dim3(128), 0,
                      s, a);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s) {
    if (a.batch == 0) return cudaSuccess;
    const int G = a.num_q_heads / a.num_kv_heads;
    if (a.head_dim == 128) return G <= 8 ? launch_cfg<128, 1, 2>(a, s) : launch_cfg<128, 2, 2>(a, s);
    return G <= 8 ? launch_cfg<64, 1, 2>(a, s) : launch_cfg<64, 2, 2>(a, s);
}

}  // namespace minisgl
