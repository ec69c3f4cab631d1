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
// Design (GB300, one CTA per SM, persistent; head_dim d = 64 or 128):
//   * Work item = (request, KV head g, block of 2*TQ new tokens), TQ =
//     floor(128/G) for any group size G = 1..16.  The block is two query
//     tiles A and B of 128 MMA rows each; row i is the (token i / G, head
//     i mod G) pair, so the G query heads that share KV head g ride in the
//     same tile and every gathered K/V tile feeds 2*128 rows (rows past
//     TQ*G, 2 at most for G in 3, 5, 6, 7, are dead: zero queries, no output).
//   * Producer warps 8-9 gather 128-token K and V tiles through page_table
//     with 16-byte cp.async into the 128-byte-swizzled layout the tensor core
//     reads (K as a K-major B operand, V as an MN-major B operand), two
//     stages deep; completion is tracked by mbarriers (cp.async.mbarrier.arrive).
//     A lane copies d/32 chunks (4 at d 128) of each of its rows, so the
//     address work per copy is small: these warps share schedulers with
//     softmax warps.
//   * Warp 11 (one lane) issues tcgen05.mma.  Per query tile X: S_X = Q_X K^T
//     (M = N = 128) into tensor memory; O_X += P_X V with P_X read from
//     tensor memory.  The issue order PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
//     keeps the tensor core on one tile while the other tile's softmax runs.
//   * Softmax warpgroups 0 (warps 0-3, tile A) and 1 (warps 4-7, tile B):
//     thread i owns TMEM lane (= MMA row) i of its tile.  It reads its S row
//     (64-column loads: maximum of the raw scores, then exponentials with
//     packed f32x2 arithmetic; in the common path the next columns' load is
//     in flight while the current ones are exponentiated), applies the causal limit C + t on diagonal
//     tiles only, keeps a running max m and sum l (base 2), and writes
//     P = 2^(s - m) as bf16 back into the upper 64 columns of its S row, where
//     the PV MMA reads it.  O_X is rescaled in tensor memory only
//     when the max has grown by more than 2^8 (the final O / l does not
//     depend on when the rescale happens).  After a query tile's first K/V
//     tile, full (unmasked) tiles skip the max pass: exponentials use the
//     running max m, P stays in registers, and only if the tile's sum shows a
//     score more than 2^20 above m (or a NaN) does the row, still intact in
//     tensor memory, go through the exact max-then-exponentiate path.  Every
//     P is then at most 2^20, well inside fp32 and bf16 range, and bf16
//     keeps the same relative precision at any magnitude.
//     Epilogue: O / l -> bf16 -> global.
//   * Tensor memory (512 columns): S_A 0-127, S_B 128-255, O_A from 256,
//     O_B from 384 (d columns each).  Shared memory: Q_A, Q_B (128 rows of
//     2d bytes each), two K/V stages (two such tiles each): 192 KB at d 128.
//   * The work-ticket counter of the dynamic schedule is the caller's when
//     given, else one of 64 library slots taken in turn.  A stream's query
//     blocks are handed out last block first (the causal limit makes it the
//     longest), so the items drawn at the end of a launch are short ones.
//   * Modes for the shared-prefix calls: prefix-only (every new token sees
//     exactly its C cached positions; fp32 rows and LSEs out), with the
//     prefix-chunk geometry computed instead of read; len_offset (a request's
//     page-table row starts past the shared positions); and a fold of an
//     fp32 partial over other positions into the bf16 output by log-sum-exp.
//   * Every mbarrier wait is bounded in time; a wait that runs out sets a
//     flag, the kernel finishes without further waiting (its output is then
//     garbage) and a device counter of such events is increased.
#include <atomic>
#include <mutex>

#include "kernels.h"
#include "tcgen05.cuh"

namespace minisgl {

__device__ unsigned int g_kernel_timeouts = 0;

// Work tickets for the extend kernel's dynamic item schedule: per call slot,
// the next ticket and the number of CTAs that have finished.  The last CTA
// of a launch puts both back to zero.
struct SchedSlot {
    unsigned int next, done;
};
__device__ SchedSlot g_sched[64];

namespace {

constexpr int ROWS = 128;                 // rows of a query tile, tokens of a KV tile
constexpr int HALF = ROWS * 128;          // one 64-column (128-byte) swizzle region of a tile
constexpr int STAGES = 2;
constexpr int RING = 8;
constexpr int SCHED_SLOTS = 64;           // per-call work-ticket counters

// Shared-memory layout for head_dim D
template <int D>
struct Smem {
    static constexpr int TILE_BYTES = ROWS * D * 2;  // 128 rows of 2D bytes
    static constexpr int OFF_Q = 0;                  // Q_A, then Q_B
    static constexpr int OFF_KV = 2 * TILE_BYTES;    // stage s: K at +2s*TILE, V at +(2s+1)*TILE
    static constexpr int OFF_BAR = OFF_KV + STAGES * 2 * TILE_BYTES;
    static constexpr int OFF_TMEM_SLOT = OFF_BAR + 192;
    static constexpr int OFF_RING = OFF_BAR + 256;   // ring of RING work-item descriptors (64 B each)
    static constexpr int OFF_PREFIX = OFF_RING + RING * 64;
};
constexpr int THREADS = 384;              // 2 softmax warpgroups, 2 producer warps, idle warp, MMA warp
constexpr int SOFTMAX_WARP0 = 0;          // warps SOFTMAX_WARP0 .. +3: tile A; +4 .. +7: tile B
constexpr int PRODUCER_WARP0 = 8;
constexpr int PRODUCER_THREADS = 64;
constexpr int PRODUCER_WARPS = 2;
// The MMA issuer is warp 11: warps are spread over the four schedulers by
// warp index mod 4, and scheduler 3 carries only softmax warps 3 and 7
// besides it (warp 10, on scheduler 2 with softmax warps 2 and 6, idles).
// A softmax warp may only touch the tensor-memory lane quarter warp % 4, so
// SOFTMAX_WARP0 must be a multiple of 4.
constexpr int MMA_WARP = 11;
static_assert(SOFTMAX_WARP0 % 4 == 0, "softmax warpgroups start on a lane-quarter boundary");
constexpr uint32_t TMEM_COLS = 512;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_LOG2 = 8.f;
constexpr long long WAIT_LIMIT = 4000000000LL;  // SM cycles (about 2 s)

__device__ __forceinline__ uint32_t col_s(int x) { return x ? 128u : 0u; }
__device__ __forceinline__ uint32_t col_o(int x) { return x ? 384u : 256u; }

// byte offset of 16-byte chunk cc (0..15) of row `row` in a 128 x 256 B tile
// stored as two 128-byte-swizzled 64-column regions
__device__ __forceinline__ uint32_t sw128(int row, int cc) {
    return (uint32_t)((cc >> 3) * HALF + (row >> 3) * 1024 + (row & 7) * 128 +
                      (((cc & 7) ^ (row & 7)) << 4));
}

// Bounded mbarrier wait shared by all roles: once one wait has run out, the
// CTA stops waiting altogether so every thread reaches the end quickly.
__device__ __forceinline__ void guarded_wait(uint32_t b, uint32_t parity, int *abort_flag) {
    if (mbar_test_wait(b, parity)) return;
    if (*((volatile int *)abort_flag)) return;
    if (!mbar_wait(b, parity, WAIT_LIMIT)) {
        *((volatile int *)abort_flag) = 1;
        atomicAdd(&g_kernel_timeouts, 1u);
    }
}

// ---- packed fp32 pairs (Blackwell f32x2 instructions) and 3-input max ----
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2split(uint64_t r, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Max of the 64 raw scores in h whose column (0..63) is <= lim (all of them
// when full).
__device__ __forceinline__ float half_max(const uint32_t (&h)[64], bool full, int lim) {
    float m0 = -INFINITY, m1 = -INFINITY;
    if (full) {
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
            m0 = fmax3(m0, __uint_as_float(h[c]), __uint_as_float(h[c + 1]));
            m1 = fmax3(m1, __uint_as_float(h[c + 2]), __uint_as_float(h[c + 3]));
        }
    } else {
#pragma unroll
        for (int c = 0; c < 64; ++c)
            if (c <= lim) m0 = fmaxf(m0, __uint_as_float(h[c]));
    }
    return fmaxf(m0, m1);
}

// P = 2^(s*scale - m) for the 32 scores in q (0 past lim unless full), added
// into the packed row sum l2 and stored as 16 bf16 pairs at TMEM column dst.
__device__ __forceinline__ void quarter_softmax(const uint32_t (&q)[32], bool full, int lim,
                                                uint64_t scale2, uint64_t negm2, uint64_t &l2,
                                                uint32_t dst) {
    uint32_t pw[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const int c = 2 * e;
        float s0 = __uint_as_float(q[c]), s1 = __uint_as_float(q[c + 1]);
        if (!full) {
            s0 = c <= lim ? s0 : -INFINITY;
            s1 = c + 1 <= lim ? s1 : -INFINITY;
        }
        float x0, x1;
        f2split(ffma2(f2(s0, s1), scale2, negm2), x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        l2 = fadd2(l2, f2(p0, p1));
        pw[e] = pack_bf16x2(p0, p1);
    }
    tmem_st16(dst, pw);
}

// 2^(s*scale - m) for the 64 scores of a full half row: 32 bf16 pairs into pw,
// sums into the packed accumulator lt
__device__ __forceinline__ void exp_half(const uint32_t (&h)[64], uint64_t scale2, uint64_t negm2,
                                         uint64_t &lt, uint32_t (&pw)[32]) {
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        float x0, x1;
        f2split(ffma2(f2(__uint_as_float(h[2 * e]), __uint_as_float(h[2 * e + 1])), scale2, negm2), x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        lt = fadd2(lt, f2(p0, p1));
        pw[e] = pack_bf16x2(p0, p1);
    }
}
// 2^(s*scale - m) for 32 scores: 16 bf16 pairs into pw[base ..]
__device__ __forceinline__ void exp_quarter(const uint32_t (&h)[32], uint64_t scale2, uint64_t negm2,
                                            uint64_t &lt, uint32_t (&pw)[32], int base) {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        float x0, x1;
        f2split(ffma2(f2(__uint_as_float(h[2 * e]), __uint_as_float(h[2 * e + 1])), scale2, negm2), x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        lt = fadd2(lt, f2(p0, p1));
        pw[base + e] = pack_bf16x2(p0, p1);
    }
}
// tcgen05.wait::ld that the compiler sees as producing r: no use of r can be
// scheduled before the wait
__device__ __forceinline__ void tmem_wait_ld_dep(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;\n"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
                   "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
                   "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
                   "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
                   "+r"(r[31])
                 :
                 : "memory");
}
// tcgen05.mma with each shared-memory descriptor given as its two 32-bit words
__device__ __forceinline__ void tc_mma_bf16_w(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                              uint32_t b_hi, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n .reg .b64 da, db;\n setp.ne.b32 p, %6, 0;\n mov.b64 da, {%1, %2};\n"
        " mov.b64 db, {%3, %4};\n tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n}\n" ::"r"(d_tmem),
        "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_mma_bf16_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                                 uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n .reg .b64 db;\n setp.ne.b32 p, %5, 0;\n mov.b64 db, {%2, %3};\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tmem_st16_from(uint32_t dst, const uint32_t (&pw)[32], int base) {
    uint32_t q[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) q[k] = pw[base + k];
    tmem_st16(dst, q);
}

__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}

// One work item: request r, KV head g, query tiles A (new tokens t0 ..
// ta_last) and B (t0 + TQ .. tb_last, when live_b), C cached tokens before
// them; nkv_a / nkv_b KV tiles seen by each tile; vis KV positions read.
struct Item {
    int r, g, t0, ta_last, tb_last, C, qoff, ooff, nkv_a, nkv_b, vis;
    bool live_b;
    __device__ __forceinline__ int nkv() const { return max(nkv_a, nkv_b); }
    __device__ __forceinline__ int n_vis() const { return vis; }
};

// Cached tokens C and new tokens E of request r: from the length arrays, or,
// for chunk r of a shared prefix (prefix_chunk_len > 0), from the chunk
// geometry: C = the chunk's length, E = the prefix_queries decode queries.
__device__ __forceinline__ void req_lens(const ExtendArgs &a, int r, int &C, int &E) {
    if (a.prefix_chunk_len > 0) {
        C = min(a.prefix_chunk_len, a.prefix_len - r * a.prefix_chunk_len);
        E = a.prefix_queries;
        return;
    }
    C = min(max(__ldg(a.cached_lens + r) - a.len_offset, 0), a.pt_width);
    // (in prefix-only mode a new token is not a page-table position)
    E = a.prefix_only ? max(__ldg(a.extend_lens + r), 0)
                      : min(max(__ldg(a.extend_lens + r), 0), a.pt_width - C);
}

// Work item `item` from the per-request prefix of item counts in shared
// memory (binary search) and the request's lengths.
__device__ __forceinline__ Item load_item(const ExtendArgs &a, const int32_t *s_prefix, int item,
                                          int TQ) {
    int lo = 0, hi = a.batch;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_prefix[mid] <= item) lo = mid; else hi = mid;
    }
    Item it;
    it.r = lo;
    const int nqb = (s_prefix[lo + 1] - s_prefix[lo]) / a.num_kv_heads;
    const int off = item - s_prefix[lo];
    it.g = off / nqb;
    // a stream's query blocks are handed out last block first: with the causal
    // limit the last block sees the most positions, so the items drawn at the
    // end of the launch (the tail) are the stream's shortest ones
    const int qb = nqb - 1 - (off - it.g * nqb);
    int E;
    req_lens(a, lo, it.C, E);
    if (a.prefix_chunk_len > 0) {  // every chunk reads q rows 0.. and writes its own rows
        it.qoff = 0;
        it.ooff = lo * a.prefix_queries;
    } else {
        it.qoff = __ldg(a.q_offsets + lo);
        it.ooff = a.out_offsets ? __ldg(a.out_offsets + lo) : it.qoff;
    }
    it.t0 = qb * 2 * TQ;
    it.ta_last = min(it.t0 + TQ, E) - 1;
    it.live_b = it.t0 + TQ < E;
    it.tb_last = it.live_b ? min(it.t0 + 2 * TQ, E) - 1 : it.ta_last;
    if (a.prefix_only) {  // every new token sees exactly the C cached positions
        it.vis = it.C;
        it.nkv_a = (it.C + ROWS - 1) / ROWS;
        it.nkv_b = it.live_b ? it.nkv_a : 0;
    } else {              // causal: token t sees C + t + 1 positions
        it.vis = it.C + it.tb_last + 1;
        it.nkv_a = (it.C + it.ta_last + 1 + ROWS - 1) / ROWS;
        it.nkv_b = it.live_b ? (it.C + it.tb_last + 1 + ROWS - 1) / ROWS : 0;
    }
    return it;
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    extend_kernel(const ExtendArgs a, const float scale_log2, const int G, const int slot) {
    using L = Smem<D>;
    constexpr int TILE_BYTES = L::TILE_BYTES;
    constexpr int OFF_Q = L::OFF_Q, OFF_KV = L::OFF_KV, OFF_BAR = L::OFF_BAR;
    constexpr int OFF_TMEM_SLOT = L::OFF_TMEM_SLOT, OFF_RING = L::OFF_RING, OFF_PREFIX = L::OFF_PREFIX;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ int s_abort;
    const uint32_t sb = smem_u32(base);
    const uint32_t sQ = sb + OFF_Q, sKV = sb + OFF_KV;
    const uint32_t bar = sb + OFF_BAR;
    auto kv_full = [&](int s) { return bar + 8 * s; };
    auto kv_empty = [&](int s) { return bar + 16 + 8 * s; };
    auto s_full = [&](int x) { return bar + 32 + 8 * x; };
    auto p_full = [&](int x) { return bar + 48 + 8 * x; };
    auto pv_done = [&](int x) { return bar + 64 + 8 * x; };
    const uint32_t fin = bar + 80, q_empty = bar + 88;
    auto item_ready = [&](uint32_t n) { return bar + 96 + 8 * (n % RING); };
    auto ring = [&](uint32_t n) { return reinterpret_cast<Item *>(base + OFF_RING + 64 * (n % RING)); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + OFF_TMEM_SLOT);
    int32_t *s_prefix = reinterpret_cast<int32_t *>(base + OFF_PREFIX);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = a.batch, Hkv = a.num_kv_heads, Hq = a.num_q_heads;
    const int TQ = ROWS / G;        // new tokens per query tile
    const int TQ2 = 2 * TQ;         // new tokens per work item
    const int live_rows = TQ * G;   // MMA rows that hold a (token, head) pair

    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(kv_full(s), PRODUCER_THREADS);
            mbar_init(kv_empty(s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(s_full(x), 1);
            mbar_init(p_full(x), 128);
            mbar_init(pv_done(x), 1);
        }
        mbar_init(fin, 1);
        mbar_init(q_empty, 1);
        for (int k = 0; k < RING; ++k) mbar_init(item_ready(k), 1);
        fence_mbar_init();
        s_abort = 0;
    }
    if (warp == MMA_WARP) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    // items per request: ceil(E / TQ2) blocks times Hkv heads, prefix in shared memory
    if (warp == PRODUCER_WARP0) {
        int carry = 0;
        if (lane == 0) s_prefix[0] = 0;
        for (int b0 = 0; b0 < B; b0 += 32) {
            const int r = b0 + lane;
            int v = 0;
            if (r < B) {
                int c, e;
                req_lens(a, r, c, e);
                v = ((e + TQ2 - 1) / TQ2) * Hkv;
                if (a.prefix_only && c == 0) v = 0;  // nothing to attend to: no items
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
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    const uint32_t idesc_pv = idesc_bf16_f32(ROWS, D, true);

    // Schedule: the CTA's first item is blockIdx.x, later ones come from a
    // ticket counter shared by the launch (items gridDim.x, gridDim.x + 1, ...
    // in the order CTAs ask), so CTAs that drew short items take more.  The
    // producers, which run ahead, draw the tickets (one item early) and
    // publish each item's description in a ring of RING slots, slot n for
    // the CTA's n-th item, with an mbarrier per slot; a description with
    // r = -1 ends the CTA's work.  A slot is rewritten RING items later, long
    // after the other roles have read it: the producers cannot get more than
    // two items ahead of the MMA warp (they wait for its q_empty), nor the MMA
    // warp more than one ahead of the softmax warps (it waits for their P).
    // The roles run through the items without a CTA-wide barrier in between;
    // each keeps its own running counts of KV tiles and of tiles per query
    // tile.
    SchedSlot *sched = a.sched ? reinterpret_cast<SchedSlot *>(a.sched) : &g_sched[slot];
    if (warp >= PRODUCER_WARP0 && warp < PRODUCER_WARP0 + PRODUCER_WARPS) {
        // ---------------- producer: Q_A, Q_B per item, then K/V tiles ----------------
        // Q tiles: thread pt copies 16-byte chunk cc of rows tb*RPT ..
        // tb*RPT+RPT-1 (d/8 threads cover one row of 2d bytes).  K/V tiles:
        // lane (rl = lane / 4, qq = lane % 4) of producer warp pw copies chunks
        // qq, qq+4, ... (d/32 of them) of tokens 16m + 8pw + rl (m = 0..7), so
        // one page-table entry and one address serve 2d/32 copies; each warp
        // instruction still writes 8 rows x 64 bytes that fall on distinct
        // banks (4 wavefronts for 512 bytes).  An item's Q goes out with its first K/V tile, once the MMA
        // warp has released the Q buffers (the previous item's last S is done).
        constexpr int CPR = D / 8;                          // 16-byte chunks per row
        constexpr int RPT = ROWS * CPR / PRODUCER_THREADS;  // Q rows per thread: 32 (d 128), 16 (d 64)
        constexpr int CI = D / 32;                          // K/V chunks a lane copies per token row
        const int pt = threadIdx.x - PRODUCER_WARP0 * 32;
        const int cc = pt % CPR, tb = pt / CPR;
        const int tok0 = (tb * RPT) / G, hh0 = (tb * RPT) - tok0 * G;  // (token, head) of row tb*RPT
        uint32_t kv_iter = 0, n_items = 0;
        int item = blockIdx.x;  // this CTA's n-th item (thread 0's copy)
        for (;; ++n_items) {
            if (pt == 0) {
                Item it;
                it.r = -1;
                if (item < total_items && !*((volatile int *)&s_abort)) it = load_item(a, s_prefix, item, TQ);
                // next ticket, drawn one item early
                if (it.r >= 0) item = (int)gridDim.x + (int)atomicAdd(&sched->next, 1u);
                *ring(n_items) = it;
                mbar_arrive(item_ready(n_items));
            }
            named_bar_sync(2, PRODUCER_THREADS);
            const Item cur = *ring(n_items);
            if (cur.r < 0) break;
            const int32_t *ptab = a.page_table + (int64_t)cur.r * a.pt_stride;
            const int n_vis = cur.n_vis(), nkv = cur.nkv();
            // lane L fetches the page-table entries of tokens (m = L/8, rl = L%8)
            // and (m = 4 + L/8, rl = L%8); the copying lanes get them by shuffle
            const int pw = pt >> 5, rl = lane >> 2, qq = lane & 3;
            auto fetch2 = [&](int j, int &ra, int &rb) {
                const int p = j * ROWS + 16 * (lane >> 3) + 8 * pw + (lane & 7);
                ra = p < n_vis ? __ldg(ptab + p) : -1;
                rb = p + 64 < n_vis ? __ldg(ptab + p + 64) : -1;
                ra = ra < 0 ? -1 : min(ra, a.num_rows - 1);
                rb = rb < 0 ? -1 : min(rb, a.num_rows - 1);
            };
            // 128-byte swizzle: chunk c of token row t sits at 16-byte slot
            // (c mod 8) xor (t mod 8); for c = qq + 4i that is one of these two
            const uint32_t xo0 = (uint32_t)((qq ^ rl) << 4), xo1 = (uint32_t)(((qq ^ rl) ^ 4) << 4);
            int ra, rb;
            fetch2(0, ra, rb);
            for (int j = 0; j < nkv; ++j) {
                const uint32_t it = kv_iter + j, st = it & 1;
                if (it >= STAGES) wait(kv_empty(st), ((it >> 1) - 1) & 1);
                if (j == 0) {
                    if (n_items > 0) wait(q_empty, (n_items - 1) & 1);
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        int tk = tok0, hd = hh0;  // (token, head) of row i, stepped along
#pragma unroll 4
                        for (int k = 0; k < RPT; ++k) {
                            const int i = tb * RPT + k;
                            const int t = cur.t0 + x * TQ + tk;
                            const bool live = i < live_rows && t <= (x ? cur.tb_last : cur.ta_last) &&
                                              (x == 0 || cur.live_b);
                            const __nv_bfloat16 *src =
                                live ? Q + ((int64_t)(cur.qoff + t) * Hq + cur.g * G + hd) * D + cc * 8 : Q;
                            cp_async_16(sQ + x * TILE_BYTES + sw128(i, cc), src, live ? 16 : 0);
                            if (++hd == G) {
                                hd = 0;
                                ++tk;
                            }
                        }
                    }
                }
                const uint32_t sK = sKV + st * 2 * TILE_BYTES, sV = sK + TILE_BYTES;
#pragma unroll
                for (int mm = 0; mm < 8; ++mm) {
                    const int row = __shfl_sync(0xffffffffu, mm < 4 ? ra : rb, ((mm & 3) << 3) | rl);
                    const int64_t e = (int64_t)max(row, 0) * a.row_stride + (int64_t)cur.g * D + qq * 8;
                    const int bytes = row >= 0 ? 16 : 0;
                    const uint32_t ob = (uint32_t)((2 * mm + pw) * 1024 + rl * 128);
#pragma unroll
                    for (int ci = 0; ci < CI; ++ci) {
                        const uint32_t o = ob + (uint32_t)((ci >> 1) * HALF) + ((ci & 1) ? xo1 : xo0);
                        cp_async_16(sK + o, Kl + e + 32 * ci, bytes);
                        cp_async_16(sV + o, Vl + e + 32 * ci, bytes);
                    }
                }
                cp_async_mbar_arrive_noinc(kv_full(st));
                // next tile's rows: the loads are in flight while this thread
                // waits for a free stage
                if (j + 1 < nkv) fetch2(j + 1, ra, rb);
            }
            kv_iter += nkv;
        }
        cp_async_wait<0>();
    } else if (warp == MMA_WARP) {
        // ---------------- MMA issuer ----------------
        // One thread (lane 0) issues every MMA, and the tensor core accepts
        // only a couple of MMAs ahead, so whatever this thread executes between
        // two MMA groups leaves the tensor core idle.  Hence: the whole warp
        // runs the bookkeeping in step, with the loop bounds and the TMEM base
        // passed through warp reductions so that every lane provably holds the
        // same value (the compiler can then keep the counters and descriptors
        // in uniform registers, which the MMA instruction reads), and only the
        // MMA and commit instructions sit under `leader`; the shared-memory
        // descriptors are built once here, and the one for K-slice kk of a
        // tile is its tile's descriptor plus a constant, added to the lower
        // 32-bit word only (the 14-bit address field holds addr >> 4, below
        // 2^14 for any shared-memory address, so the sum never carries into
        // the next field, and the upper word is the same for every Q and K
        // tile, and for every V tile); and a wait first probes
        // the barrier once, taking the bounded, abort-aware path only when
        // the phase is not complete yet.
        {
            const bool leader = lane == 0;
            // the TMEM base is the same in every lane; a warp reduction makes
            // that visible to the compiler
            const uint32_t tm = __reduce_max_sync(0xffffffffu, tmem);
            const uint64_t dq0 = smem_desc_sw128(sQ, 16, 1024);
            const uint64_t dq1 = smem_desc_sw128(sQ + TILE_BYTES, 16, 1024);
            const uint64_t dk0 = smem_desc_sw128(sKV, 16, 1024);
            const uint64_t dk1 = smem_desc_sw128(sKV + 2 * TILE_BYTES, 16, 1024);
            const uint64_t dv0 = smem_desc_sw128(sKV + TILE_BYTES, HALF, 1024);
            const uint64_t dv1 = smem_desc_sw128(sKV + 3 * TILE_BYTES, HALF, 1024);
            auto mwait = [&](uint32_t b, uint32_t par) {
                if (!mbar_test_wait(b, par)) wait(b, par);
            };
            uint32_t kv_iter = 0, cnt_a = 0, cnt_b = 0;
            for (uint32_t n = 0;; ++n) {
                wait(item_ready(n), (n / RING) & 1);
                const Item cur = *ring(n);
                const unsigned stop = (*((volatile int *)&s_abort) || cur.r < 0) ? 1u : 0u;
                if (__reduce_max_sync(0xffffffffu, stop)) break;
                const int nkv_a = (int)__reduce_max_sync(0xffffffffu, (unsigned)cur.nkv_a);
                const int nkv_b = (int)__reduce_max_sync(0xffffffffu, (unsigned)cur.nkv_b);
                const int nkv = max(nkv_a, nkv_b);
                const uint32_t dhi = (uint32_t)(dq0 >> 32);  // same upper word for every Q/K descriptor
                const uint32_t vhi = (uint32_t)(dv0 >> 32);
                auto issue_s = [&](int x, int j) {  // S_X(j) = Q_X K(j)^T
                    const uint32_t dk = (uint32_t)(((kv_iter + j) & 1) ? dk1 : dk0);
                    const uint32_t dq = (uint32_t)(x ? dq1 : dq0);
                    const uint32_t ds = tm + col_s(x);
                    if (leader) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            // K-slice kk of a K-major 128-byte-swizzled tile: 64-column
                            // region kk / 4, 32-byte step kk % 4 within the row
                            const uint32_t off = (uint32_t)(((kk >> 2) * HALF + (kk & 3) * 32) >> 4);
                            tc_mma_bf16_w(ds, dq + off, dhi, dk + off, dhi, idesc_qk, kk > 0 ? 1u : 0u);
                        }
                        tc_commit(s_full(x));
                    }
                };
                auto issue_pv = [&](int x, int j, uint32_t cnt) {  // O_X += P_X(j) V(j)
                    mwait(p_full(x), (cnt + j) & 1);
                    tc_fence_after();
                    const uint32_t dv = (uint32_t)(((kv_iter + j) & 1) ? dv1 : dv0);
                    const uint32_t dO = tm + col_o(x), dP = tm + col_s(x) + 64;
                    if (leader) {
#pragma unroll
                        for (int kk = 0; kk < ROWS / 16; ++kk)  // 16 tokens (2 KB of V) per MMA
                            tc_mma_bf16_ts_w(dO, dP + kk * 8, dv + (uint32_t)(kk * (2048 >> 4)), vhi,
                                             idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                        tc_commit(pv_done(x));
                    }
                };
                auto wait_kv = [&](int j) {
                    mwait(kv_full((kv_iter + j) & 1), ((kv_iter + j) >> 1) & 1);
                    fence_proxy_async_smem();
                    tc_fence_after();
                };
                // The first S of each tile of this item reads Q_A / Q_B; once the
                // last of them is issued, q_empty (fired when they are done)
                // lets the producers bring in the next item's Q.
                wait_kv(0);
                issue_s(0, 0);
                if (nkv_b > 0) issue_s(1, 0);
                if (nkv == 1 && leader) tc_commit(q_empty);
                for (int j = 0; j < nkv; ++j) {
                    bool next_ready = false;
                    if (j < nkv_a) issue_pv(0, j, cnt_a);
                    if (j + 1 < nkv_a) {
                        wait_kv(j + 1);
                        next_ready = true;
                        issue_s(0, j + 1);
                    }
                    if (j < nkv_b) issue_pv(1, j, cnt_b);
                    // every MMA reading this stage is issued
                    if (leader) tc_commit(kv_empty((kv_iter + j) & 1));
                    if (j + 1 < nkv_b) {
                        if (!next_ready) wait_kv(j + 1);
                        issue_s(1, j + 1);
                    }
                    if (j + 2 == nkv && leader) tc_commit(q_empty);
                }
                kv_iter += nkv;
                cnt_a += nkv_a;
                cnt_b += nkv_b;
            }
        }
        __syncwarp();
    } else if (warp >= SOFTMAX_WARP0 && warp < SOFTMAX_WARP0 + 8) {
        // ---------------- softmax / epilogue: thread i owns row i of tile x ----------------
        // O_X is read out before this warpgroup publishes the next item's
        // first P_X, and the MMA that overwrites O_X (that item's first PV_X)
        // waits for that P_X.
        const int x = (warp - SOFTMAX_WARP0) >> 2;
        const int i = threadIdx.x - SOFTMAX_WARP0 * 32 - x * 128;
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t scol = lane_base + col_s(x), ocol = lane_base + col_o(x);
        const uint64_t scale2 = f2(scale_log2, scale_log2);
        uint32_t cnt = 0;  // tiles of query tile x processed
        for (uint32_t n = 0;; ++n) {
            wait(item_ready(n), (n / RING) & 1);
            if (*((volatile int *)&s_abort)) break;
            const Item cur = *ring(n);
            if (cur.r < 0) break;
            const int nkv_x = x ? cur.nkv_b : cur.nkv_a;
            if (nkv_x > 0) {
                const int t_last = x ? cur.tb_last : cur.ta_last;
                const int tt = cur.t0 + x * TQ + i / G;
                const bool live = i < live_rows && tt <= t_last;
                const int t = min(tt, t_last);
                const int lim = a.prefix_only ? cur.C - 1 : cur.C + t;  // last visible position
                float m = -INFINITY;            // running max of scaled scores (base 2)
                uint64_t l2 = f2(0.f, 0.f);     // running row sum, two partial lanes
                for (int j = 0; j < nkv_x; ++j) {
                    wait(s_full(x), (cnt + j) & 1);
                    tc_fence_after();
                    const int rel = lim - j * ROWS;  // last visible column of this tile
                    const bool full = rel >= ROWS - 1;
                    if (j > 0 && __all_sync(0xffffffffu, full)) {
                        // Running-max fast path: exponentials with the max m of the
                        // earlier tiles, no max pass.  P stays in registers until the
                        // tile's sum shows no score exceeded m by more than 20 (base
                        // 2); otherwise (or on NaN) the S row, still intact, goes
                        // through the exact path below.
                        const uint64_t negm2 = f2(-m, -m);
                        uint32_t p0[32], p1[32];
                        uint64_t lt = f2(0.f, 0.f);
                        {
                            // the second half's loads are in flight while the
                            // previous part's exponentials run
                            uint32_t h[64], c2[32], c3[32];
                            tmem_ld64(scol, h);
                            tmem_wait_ld();
                            tmem_ld32(scol + 64, c2);
                            exp_half(h, scale2, negm2, lt, p0);
                            tmem_wait_ld_dep(c2);
                            tmem_ld32(scol + 96, c3);
                            exp_quarter(c2, scale2, negm2, lt, p1, 0);
                            tmem_wait_ld_dep(c3);
                            exp_quarter(c3, scale2, negm2, lt, p1, 16);
                        }
                        float ta, tb;
                        f2split(lt, ta, tb);
                        const float ts = ta + tb;
                        if (!__any_sync(0xffffffffu, !(ts <= 1048576.f))) {
                            tmem_st16_from(scol + 64, p0, 0);
                            tmem_st16_from(scol + 80, p0, 16);
                            tmem_st16_from(scol + 96, p1, 0);
                            tmem_st16_from(scol + 112, p1, 16);
                            l2 = fadd2(l2, lt);
                            tmem_wait_st();
                            tc_fence_before();
                            mbar_arrive(p_full(x));
                            continue;
                        }
                    }
                    // pass 1: max of the raw scores (sm_scale > 0); the last 32
                    // columns stay in registers for pass 2
                    uint32_t top[32];
                    float mx;
                    {
                        uint32_t h[64];
                        tmem_ld64(scol, h);
                        tmem_wait_ld();
                        mx = half_max(h, full, rel);
                        tmem_ld64(scol + 64, h);
                        tmem_wait_ld();
                        mx = fmaxf(mx, half_max(h, full, rel - 64));
#pragma unroll
                        for (int c = 0; c < 32; ++c) top[c] = h[32 + c];
                    }
                    const float m_new = fmaxf(m, mx * scale_log2);
                    if (j > 0) {
                        wait(pv_done(x), (cnt + j - 1) & 1);  // PV(j-1) done: O settled
                        tc_fence_after();
                        if (__any_sync(0xffffffffu, m_new > m + RESCALE_LOG2)) {
                            const float alpha = ex2(m - m_new);
                            float la, lb;
                            f2split(l2, la, lb);
                            l2 = f2(la * alpha, lb * alpha);
                            m = m_new;
#pragma unroll 1
                            for (int q4 = 0; q4 < D / 32; ++q4) {
                                uint32_t o[32];
                                tmem_ld32(ocol + 32 * q4, o);
                                tmem_wait_ld();
#pragma unroll
                                for (int c = 0; c < 32; ++c)
                                    o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                                tmem_st32(ocol + 32 * q4, o);
                            }
                        }
                    } else {
                        m = m_new;
                    }
                    // pass 2: P as bf16 into the upper 64 columns of this S row,
                    // quarter by quarter from the top: S columns 32q..32q+31 ->
                    // P columns 64+16q..64+16q+15, which only ever overwrites S
                    // columns already consumed
                    const uint64_t negm2 = f2(-m, -m);
                    quarter_softmax(top, full, rel - 96, scale2, negm2, l2, scol + 112);
#pragma unroll 1
                    for (int q4 = 2; q4 >= 0; --q4) {
                        uint32_t qv[32];
                        tmem_ld32(scol + 32 * q4, qv);
                        tmem_wait_ld();
                        quarter_softmax(qv, full, rel - 32 * q4, scale2, negm2, l2, scol + 64 + 16 * q4);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(p_full(x));
                }
                float la, lb;
                f2split(l2, la, lb);
                const float l = la + lb;
                // epilogue: O / l -> bf16
                wait(pv_done(x), (cnt + nkv_x - 1) & 1);
                tc_fence_after();
                float inv = 1.f / l;
                const int64_t orow = (int64_t)(cur.ooff + t) * Hq + cur.g * G + (i % G);
                // with a partial over other positions to fold in: out = (w_s o/l + w_p o_p) / (w_s + w_p),
                // w = 2^(lse - max) in base 2 (this row's lse is m + log2 l)
                float cp = 0.f;
                const float *mrow = nullptr;
                if (a.merge_o && live) {
                    const float ls = m + log2f(l), lp = a.merge_lse[orow] * LOG2E;
                    const float mx = fmaxf(ls, lp);
                    const float ws = ex2(ls - mx), wp = ex2(lp - mx);
                    const float it = 1.f / (ws + wp);
                    inv *= ws * it;
                    cp = wp * it;
                    mrow = a.merge_o + orow * D;
                }
                __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) + orow * D;
                if (a.out_f32 && live)  // natural-log LSE of the scaled scores
                    a.lse_out[orow] = (m + log2f(l)) * 0.6931471805599453f;
#pragma unroll 1
                for (int q4 = 0; q4 < D / 32; ++q4) {
                    uint32_t o[32];
                    tmem_ld32(ocol + 32 * q4, o);
                    tmem_wait_ld();
                    if (a.out_f32) {  // normalised fp32 rows for a later merge
                        if (live) {
                            float *fd = a.out_f32 + orow * D + 32 * q4;
#pragma unroll
                            for (int c = 0; c < 32; c += 4)
                                *reinterpret_cast<float4 *>(fd + c) =
                                    make_float4(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv,
                                                __uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
                        }
                    } else if (mrow) {
#pragma unroll
                        for (int c = 0; c < 32; c += 8) {
                            const float4 p0 = *reinterpret_cast<const float4 *>(mrow + 32 * q4 + c);
                            const float4 p1 = *reinterpret_cast<const float4 *>(mrow + 32 * q4 + c + 4);
                            uint4 v;
                            v.x = pack_bf16x2(__uint_as_float(o[c + 0]) * inv + cp * p0.x,
                                              __uint_as_float(o[c + 1]) * inv + cp * p0.y);
                            v.y = pack_bf16x2(__uint_as_float(o[c + 2]) * inv + cp * p0.z,
                                              __uint_as_float(o[c + 3]) * inv + cp * p0.w);
                            v.z = pack_bf16x2(__uint_as_float(o[c + 4]) * inv + cp * p1.x,
                                              __uint_as_float(o[c + 5]) * inv + cp * p1.y);
                            v.w = pack_bf16x2(__uint_as_float(o[c + 6]) * inv + cp * p1.z,
                                              __uint_as_float(o[c + 7]) * inv + cp * p1.w);
                            *reinterpret_cast<uint4 *>(dst + 32 * q4 + c) = v;
                        }
                    } else if (live) {
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
                cnt += nkv_x;
            }
        }
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
    // the last CTA to finish leaves the ticket counter at zero for the next
    // launch that uses this slot (a launch in the same stream starts drawing
    // only after this grid has completed)
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&sched->done, 1u) == gridDim.x - 1) {
            sched->next = 0;
            sched->done = 0;
            __threadfence();
        }
    }
}

namespace {

// Raise the kernel's dynamic shared-memory limit once per device.
template <int D>
cudaError_t configure_extend() {
    static std::mutex mu;
    static bool configured[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(extend_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Smem<D>::OFF_PREFIX + 4097 * 4 + 1024);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return e;
        }
        configured[dev] = true;
    }
    return cudaSuccess;
}

template <int D>
cudaError_t launch_extend_d(const ExtendArgs &a, cudaStream_t s, int grid) {
    if (cudaError_t e = configure_extend<D>()) return e;
    const int G = a.num_q_heads / a.num_kv_heads;
    const size_t smem = (size_t)Smem<D>::OFF_PREFIX + (size_t)(a.batch + 1) * 4 + 1024;
    // without a caller counter, a library ticket-counter slot per call, so
    // calls running at the same time on different streams do not share one
    static std::atomic<unsigned> next_slot{0};
    const int slot = a.sched ? 0 : (int)(next_slot.fetch_add(1u) % SCHED_SLOTS);
    return launch_pdl(extend_kernel<D>, dim3((unsigned)grid), dim3(THREADS), smem, s, a,
                      a.sm_scale * LOG2E, G, slot);
}

}  // namespace

int extend_grid(const ExtendArgs &a) {
    const int G = a.num_q_heads / a.num_kv_heads;
    const int TQ2 = 2 * (ROWS / G);
    // work items: exact for prefix chunks (every chunk has all the queries),
    // else an upper bound (every request can add one partial block)
    const int64_t items = a.prefix_chunk_len > 0
                              ? (int64_t)a.batch * ((a.prefix_queries + TQ2 - 1) / TQ2) * a.num_kv_heads
                              : ((int64_t)a.total_q_tokens / TQ2 + a.batch) * a.num_kv_heads;
    int64_t grid = device_sm_count();
    if (grid > items) grid = items;
    if (grid < 1) grid = 1;
    return (int)grid;
}

cudaError_t launch_extend(const ExtendArgs &a, cudaStream_t s) {
    if (a.batch == 0 || a.total_q_tokens == 0) return cudaSuccess;
    const int grid = extend_grid(a);
    return a.head_dim == 64 ? launch_extend_d<64>(a, s, grid) : launch_extend_d<128>(a, s, grid);
}

cudaError_t read_kernel_timeouts(unsigned int *count) {
    return cudaMemcpyFromSymbol(count, g_kernel_timeouts, sizeof(unsigned int));
}

}  // namespace minisgl
