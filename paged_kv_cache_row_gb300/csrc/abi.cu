// abi.cu -- the extern "C" entry points declared in include/minisgl.h.
//
// Host-side argument checks, the thread-local error string, workspace
// carving, and the launches.  No entry point allocates device memory or
// synchronises with the device.
#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>

#include <nvtx3/nvToolsExt.h>

#include "kernels.h"
#include "minisgl.h"

namespace {

thread_local std::string g_err;

// An NVTX range around each entry point, so a profiler timeline shows the
// library's calls by name (NVTX does nothing unless a tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_pool(const minisgl_kv_pool *p, int32_t layer, const char *who) {
    if (!p) return fail(MINISGL_ERR_ARG, "%s: pool descriptor is NULL", who);
    if (p->dtype != MINISGL_BF16) return fail(MINISGL_ERR_DTYPE, "%s: pool dtype must be bf16", who);
    if (!p->k_base || !p->v_base) return fail(MINISGL_ERR_ARG, "%s: pool base is NULL", who);
    if (p->head_dim != 64 && p->head_dim != 128)
        return fail(MINISGL_ERR_UNSUPPORTED, "%s: head_dim %d not in {64, 128}", who, p->head_dim);
    if (p->num_kv_heads < 1 || p->num_rows < 1 || p->num_layers < 1)
        return fail(MINISGL_ERR_SHAPE, "%s: pool sizes must be positive", who);
    if (p->row_stride < (int64_t)p->num_kv_heads * p->head_dim || p->row_stride % 8 != 0)
        return fail(MINISGL_ERR_SHAPE, "%s: row_stride %lld must be >= H_kv*d and a multiple of 8",
                    who, (long long)p->row_stride);
    if (p->layer_stride % 8 != 0 || p->layer_stride < 0)
        return fail(MINISGL_ERR_SHAPE, "%s: layer_stride must be a non-negative multiple of 8", who);
    if (!aligned16(p->k_base) || !aligned16(p->v_base))
        return fail(MINISGL_ERR_SHAPE, "%s: pool bases must be 16-byte aligned", who);
    if (layer < 0 || layer >= p->num_layers)
        return fail(MINISGL_ERR_ARG, "%s: layer %d outside [0, %d)", who, layer, p->num_layers);
    return MINISGL_OK;
}

const void *layer_ptr(const void *base, const minisgl_kv_pool *p, int32_t layer) {
    return static_cast<const char *>(base) + (size_t)layer * p->layer_stride * 2;
}

int cuda_status(cudaError_t e, const char *who) {
    if (e == cudaSuccess) return MINISGL_OK;
    return fail(MINISGL_ERR_CUDA, "%s: %s", who, cudaGetErrorString(e));
}

constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t ws_bytes(int64_t batch, int64_t hq, int64_t hkv, int64_t d, int64_t splits) {
    return align256(batch * hkv * 4) + align256(batch * hq * splits * 4) + batch * hq * splits * d * 4;
}

int check_heads(int32_t hq, int32_t hkv, int max_group, const char *who) {
    if (hq < 1 || hq % hkv != 0)
        return fail(MINISGL_ERR_SHAPE, "%s: num_q_heads %d is not a multiple of num_kv_heads %d",
                    who, hq, hkv);
    if (hq / hkv > max_group)
        return fail(MINISGL_ERR_UNSUPPORTED, "%s: group size %d > %d", who, hq / hkv, max_group);
    return MINISGL_OK;
}

}  // namespace

namespace minisgl {
namespace {
std::atomic<int> g_pdl{-1};  // -1: not read from the environment yet
}
bool pdl_enabled() {
    int v = g_pdl.load(std::memory_order_relaxed);
    if (v < 0) {
        const char *e = std::getenv("MINISGL_PDL");
        v = (e && e[0] == '0' && e[1] == '\0') ? 0 : 1;
        int expect = -1;
        if (!g_pdl.compare_exchange_strong(expect, v)) v = expect;
    }
    return v != 0;
}

int report_error(int code, const char *msg) {
    g_err = msg;
    return code;
}

int device_sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = n;
    }
    return cached[dev];
}
}  // namespace minisgl

extern "C" {

const char *minisgl_last_error(void) { return g_err.c_str(); }

int32_t minisgl_device_sm_count(void) { return minisgl::device_sm_count(); }

int minisgl_debug_set_pdl(int enabled) {
    const int prev = minisgl::pdl_enabled() ? 1 : 0;
    minisgl::g_pdl.store(enabled ? 1 : 0);
    return prev;
}

int minisgl_debug_timeout_count(uint32_t *count) {
    g_err.clear();
    if (!count) return fail(MINISGL_ERR_ARG, "debug_timeout_count: NULL count");
    unsigned int c = 0;
    if (int rc = cuda_status(minisgl::read_kernel_timeouts(&c), "debug_timeout_count")) return rc;
    *count = c;
    return MINISGL_OK;
}

int minisgl_store_kv(const minisgl_kv_pool *pool, int32_t layer, const void *k, const void *v,
                     int64_t k_tok_stride, int64_t v_tok_stride, const int32_t *out_loc,
                     int32_t n_tokens, void *stream) {
    g_err.clear();
    NvtxRange nvtx_range("minisgl_store_kv");
    if (int rc = check_pool(pool, layer, "store_kv")) return rc;
    if (n_tokens < 0) return fail(MINISGL_ERR_ARG, "store_kv: n_tokens < 0");
    if (n_tokens == 0) return MINISGL_OK;
    if (!k || !v || !out_loc) return fail(MINISGL_ERR_ARG, "store_kv: NULL k, v or out_loc");
    const int64_t row = (int64_t)pool->num_kv_heads * pool->head_dim;
    if (!aligned16(k) || !aligned16(v))
        return fail(MINISGL_ERR_SHAPE, "store_kv: k and v must be 16-byte aligned");
    if (k_tok_stride < row || v_tok_stride < row || k_tok_stride % 8 || v_tok_stride % 8)
        return fail(MINISGL_ERR_SHAPE, "store_kv: token strides must be >= H_kv*d and multiples of 8");
    if ((int64_t)n_tokens * (row / 4) >= (int64_t(1) << 31))
        return fail(MINISGL_ERR_UNSUPPORTED, "store_kv: n_tokens * H_kv * d too large for one call");
    minisgl::StoreArgs a;
    a.k_layer = const_cast<void *>(layer_ptr(pool->k_base, pool, layer));
    a.v_layer = const_cast<void *>(layer_ptr(pool->v_base, pool, layer));
    a.row_stride = pool->row_stride;
    a.num_rows = pool->num_rows;
    a.k = k;
    a.v = v;
    a.k_tok_stride = k_tok_stride;
    a.v_tok_stride = v_tok_stride;
    a.out_loc = out_loc;
    a.n_tokens = n_tokens;
    a.row_elems = (int32_t)row;
    return cuda_status(minisgl::launch_store_kv(a, static_cast<cudaStream_t>(stream)), "store_kv");
}

size_t minisgl_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t max_splits) {
    if (batch < 0 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 || max_splits < 2 ||
        max_splits > 256)
        return 0;
    return ws_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_splits);
}

}  // extern "C"

namespace {

// The new K/V rows of minisgl_store_decode_attn (null for plain decode).
struct FusedStore {
    const void *k, *v;
    int64_t k_tok_stride, v_tok_stride;
    const int32_t *out_loc;
};

int decode_impl(const minisgl_kv_pool *pool, int32_t layer, const void *q, int32_t num_q_heads,
                const int32_t *page_table, int32_t batch, int64_t pt_row_stride, int32_t pt_width,
                const int32_t *seq_lens, float sm_scale, void *out, void *workspace,
                size_t workspace_bytes, int32_t split_tokens, void *stream, const FusedStore *fs) {
    if (int rc = check_pool(pool, layer, "decode_attn")) return rc;
    if (int rc = check_heads(num_q_heads, pool->num_kv_heads, 16, "decode_attn")) return rc;
    if (batch < 0 || batch > 4096) return fail(MINISGL_ERR_ARG, "decode_attn: batch %d outside [0, 4096]", batch);
    if (batch == 0) return MINISGL_OK;
    if (!q || !page_table || !seq_lens || !out)
        return fail(MINISGL_ERR_ARG, "decode_attn: NULL q, page_table, seq_lens or out");
    if (!aligned16(q) || !aligned16(out))
        return fail(MINISGL_ERR_SHAPE, "decode_attn: q and out must be 16-byte aligned");
    if (pt_width < 0 || pt_row_stride < pt_width)
        return fail(MINISGL_ERR_SHAPE, "decode_attn: need 0 <= pt_width <= pt_row_stride");
    if (split_tokens < 0) return fail(MINISGL_ERR_ARG, "decode_attn: split_tokens < 0");
    const int64_t tiles = (int64_t)batch * pool->num_kv_heads * ((pt_width + 15) / 16);
    if (tiles >= (int64_t(1) << 31))
        return fail(MINISGL_ERR_UNSUPPORTED, "decode_attn: batch * H_kv * width too large");
    // the largest split count the workspace holds
    int splits = 0;
    if (workspace && ((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0)) {
        for (int s = 256; s >= 2; --s)
            if (ws_bytes(batch, num_q_heads, pool->num_kv_heads, pool->head_dim, s) <= workspace_bytes) {
                splits = s;
                break;
            }
    }
    if (splits < 2)
        return fail(MINISGL_ERR_WORKSPACE,
                    "decode_attn: workspace must be 256-byte aligned and hold >= 2 splits (%zu bytes)",
                    ws_bytes(batch, num_q_heads, pool->num_kv_heads, pool->head_dim, 2));
    minisgl::DecodeArgs a;
    a.q = q;
    a.k_layer = layer_ptr(pool->k_base, pool, layer);
    a.v_layer = layer_ptr(pool->v_base, pool, layer);
    a.row_stride = pool->row_stride;
    a.num_rows = pool->num_rows;
    a.page_table = page_table;
    a.pt_stride = pt_row_stride;
    a.pt_width = pt_width;
    a.seq_lens = seq_lens;
    a.batch = batch;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = pool->num_kv_heads;
    a.head_dim = pool->head_dim;
    a.sm_scale = sm_scale;
    a.out = out;
    char *ws = static_cast<char *>(workspace);
    a.split_count = reinterpret_cast<int32_t *>(ws);
    ws += align256((size_t)batch * pool->num_kv_heads * 4);
    a.ws_lse = reinterpret_cast<float *>(ws);
    ws += align256((size_t)batch * num_q_heads * splits * 4);
    a.ws_o = reinterpret_cast<float *>(ws);
    a.max_splits = splits;
    a.split_tokens = split_tokens;
    a.lse_out = nullptr;
    a.out_loc = fs ? fs->out_loc : nullptr;
    a.k_new = fs ? fs->k : nullptr;
    a.v_new = fs ? fs->v : nullptr;
    a.new_k_stride = fs ? fs->k_tok_stride : 0;
    a.new_v_stride = fs ? fs->v_tok_stride : 0;
    return cuda_status(minisgl::launch_decode(a, static_cast<cudaStream_t>(stream)), "decode_attn");
}

}  // namespace

extern "C" {

int minisgl_decode_attn(const minisgl_kv_pool *pool, int32_t layer, const void *q,
                        int32_t num_q_heads, const int32_t *page_table, int32_t batch,
                        int64_t pt_row_stride, int32_t pt_width, const int32_t *seq_lens,
                        float sm_scale, void *out, void *workspace, size_t workspace_bytes,
                        int32_t split_tokens, void *stream) {
    g_err.clear();
    NvtxRange nvtx_range("minisgl_decode_attn");
    return decode_impl(pool, layer, q, num_q_heads, page_table, batch, pt_row_stride, pt_width,
                       seq_lens, sm_scale, out, workspace, workspace_bytes, split_tokens, stream,
                       nullptr);
}

int minisgl_store_decode_attn(const minisgl_kv_pool *pool, int32_t layer, const void *k,
                              const void *v, int64_t k_tok_stride, int64_t v_tok_stride,
                              const int32_t *out_loc, const void *q, int32_t num_q_heads,
                              const int32_t *page_table, int32_t batch, int64_t pt_row_stride,
                              int32_t pt_width, const int32_t *seq_lens, float sm_scale, void *out,
                              void *workspace, size_t workspace_bytes, int32_t split_tokens,
                              void *stream) {
    g_err.clear();
    NvtxRange nvtx_range("minisgl_store_decode_attn");
    if (int rc = check_pool(pool, layer, "store_decode_attn")) return rc;
    if (batch > 0) {
        if (!k || !v || !out_loc) return fail(MINISGL_ERR_ARG, "store_decode_attn: NULL k, v or out_loc");
        const int64_t row = (int64_t)pool->num_kv_heads * pool->head_dim;
        if (!aligned16(k) || !aligned16(v))
            return fail(MINISGL_ERR_SHAPE, "store_decode_attn: k and v must be 16-byte aligned");
        if (k_tok_stride < row || v_tok_stride < row || k_tok_stride % 8 || v_tok_stride % 8)
            return fail(MINISGL_ERR_SHAPE,
                        "store_decode_attn: token strides must be >= H_kv*d and multiples of 8");
    }
    const FusedStore fs{k, v, k_tok_stride, v_tok_stride, out_loc};
    return decode_impl(pool, layer, q, num_q_heads, page_table, batch, pt_row_stride, pt_width,
                       seq_lens, sm_scale, out, workspace, workspace_bytes, split_tokens, stream, &fs);
}

int minisgl_extend_attn(const minisgl_kv_pool *pool, int32_t layer, const void *q,
                        int32_t num_q_heads, const int32_t *page_table, int32_t batch,
                        int64_t pt_row_stride, int32_t pt_width, const int32_t *cached_lens,
                        const int32_t *extend_lens, const int32_t *q_offsets,
                        int32_t total_q_tokens, float sm_scale, void *out, uint32_t *work_counter,
                        void *stream) {
    g_err.clear();
    NvtxRange nvtx_range("minisgl_extend_attn");
    if (int rc = check_pool(pool, layer, "extend_attn")) return rc;
    if (int rc = check_heads(num_q_heads, pool->num_kv_heads, 16, "extend_attn")) return rc;
    if (work_counter && (reinterpret_cast<uintptr_t>(work_counter) & 7u))
        return fail(MINISGL_ERR_ARG, "extend_attn: work_counter must be 8-byte aligned");
    if (batch < 0 || batch > 4096) return fail(MINISGL_ERR_ARG, "extend_attn: batch %d outside [0, 4096]", batch);
    if (total_q_tokens < 0) return fail(MINISGL_ERR_ARG, "extend_attn: total_q_tokens < 0");
    if (!(sm_scale > 0.f) || !(sm_scale < 3.0e38f))
        return fail(MINISGL_ERR_ARG, "extend_attn: sm_scale must be positive and finite");
    if (batch == 0 || total_q_tokens == 0) return MINISGL_OK;
    if (!q || !page_table || !cached_lens || !extend_lens || !q_offsets || !out)
        return fail(MINISGL_ERR_ARG, "extend_attn: NULL pointer argument");
    if (!aligned16(q) || !aligned16(out))
        return fail(MINISGL_ERR_SHAPE, "extend_attn: q and out must be 16-byte aligned");
    if (pt_width < 0 || pt_row_stride < pt_width)
        return fail(MINISGL_ERR_SHAPE, "extend_attn: need 0 <= pt_width <= pt_row_stride");
    minisgl::ExtendArgs a;
    a.q = q;
    a.k_layer = layer_ptr(pool->k_base, pool, layer);
    a.v_layer = layer_ptr(pool->v_base, pool, layer);
    a.row_stride = pool->row_stride;
    a.num_rows = pool->num_rows;
    a.page_table = page_table;
    a.pt_stride = pt_row_stride;
    a.pt_width = pt_width;
    a.cached_lens = cached_lens;
    a.extend_lens = extend_lens;
    a.q_offsets = q_offsets;
    a.batch = batch;
    a.total_q_tokens = total_q_tokens;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = pool->num_kv_heads;
    a.head_dim = pool->head_dim;
    a.sm_scale = sm_scale;
    a.out = out;
    a.prefix_only = 0;
    a.out_f32 = nullptr;
    a.lse_out = nullptr;
    a.out_offsets = nullptr;
    a.sched = work_counter;
    return cuda_status(minisgl::launch_extend(a, static_cast<cudaStream_t>(stream)), "extend_attn");
}

}  // extern "C"

namespace {

constexpr int CASCADE_MAX_CHUNKS = 32;

constexpr int CASCADE_SUFFIX_SPLITS = 16;  // the merge kernel holds at most 16 suffix splits

// Workspace layout of minisgl_cascade_decode_attn (each part 256-byte aligned):
// the prefix launch's work-ticket counter (8 bytes in a 256-byte part), fp32
// prefix partials [chunks, B, Hq, D] and their LSEs [chunks, B, Hq], then a
// decode workspace for the suffix's split partials.
// Most prefix chunks a call with this shape uses: about two work items per
// SM (a work item covers 2*floor(128/G) query tokens of one KV head), at
// most 32.
int64_t cascade_chunk_cap(int64_t batch, int64_t hq, int64_t hkv) {
    const int64_t g = std::max<int64_t>(1, hq / hkv);
    const int64_t tq2 = std::max<int64_t>(1, 2 * (128 / g));
    const int64_t items = std::max<int64_t>(1, ((batch + tq2 - 1) / tq2) * hkv);
    int64_t sms = minisgl::device_sm_count();
    if (sms <= 0) sms = 1024;  // no device: the 32-chunk ceiling decides
    return std::max<int64_t>(1, std::min<int64_t>((2 * sms + items - 1) / items, CASCADE_MAX_CHUNKS));
}

size_t cascade_bytes(int64_t batch, int64_t hq, int64_t hkv, int64_t d, int64_t chunks) {
    return 256 + align256((size_t)chunks * batch * hq * d * 4) + align256((size_t)chunks * batch * hq * 4) +
           ws_bytes(batch, hq, hkv, d, CASCADE_SUFFIX_SPLITS);
}

}  // namespace

extern "C" {

size_t minisgl_cascade_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim) {
    if (batch < 0 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1) return 0;
    return cascade_bytes(batch, num_q_heads, num_kv_heads, head_dim,
                         cascade_chunk_cap(batch, num_q_heads, num_kv_heads));
}

int minisgl_cascade_decode_attn(const minisgl_kv_pool *pool, int32_t layer, const void *q,
                                int32_t num_q_heads, const int32_t *page_table, int32_t batch,
                                int64_t pt_row_stride, int32_t pt_width, const int32_t *seq_lens,
                                int32_t shared_len, float sm_scale, void *out, void *workspace,
                                size_t workspace_bytes, void *stream) {
    g_err.clear();
    NvtxRange nvtx_range("minisgl_cascade_decode_attn");
    if (int rc = check_pool(pool, layer, "cascade_decode_attn")) return rc;
    if (int rc = check_heads(num_q_heads, pool->num_kv_heads, 16, "cascade_decode_attn")) return rc;
    if (batch < 0 || batch > 4096)
        return fail(MINISGL_ERR_ARG, "cascade_decode_attn: batch %d outside [0, 4096]", batch);
    if (!(sm_scale > 0.f) || !(sm_scale < 3.0e38f))
        return fail(MINISGL_ERR_ARG, "cascade_decode_attn: sm_scale must be positive and finite");
    if (pt_width < 1 || pt_row_stride < pt_width)
        return fail(MINISGL_ERR_SHAPE, "cascade_decode_attn: need 1 <= pt_width <= pt_row_stride");
    if (shared_len < 1 || shared_len > pt_width)
        return fail(MINISGL_ERR_ARG, "cascade_decode_attn: shared_len %d outside [1, pt_width]", shared_len);
    if (batch == 0) return MINISGL_OK;
    if (!q || !page_table || !seq_lens || !out || !workspace)
        return fail(MINISGL_ERR_ARG, "cascade_decode_attn: NULL pointer argument");
    if (!aligned16(q) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(MINISGL_ERR_SHAPE, "cascade_decode_attn: q, out 16-byte and workspace 256-byte aligned");
    // prefix chunks: about two work items per SM, at least four 128-token tiles each
    const int64_t tiles = (shared_len + 127) / 128;
    int64_t chunks = cascade_chunk_cap(batch, num_q_heads, pool->num_kv_heads);
    chunks = std::max<int64_t>(1, std::min<int64_t>(chunks, (tiles + 3) / 4));
    const int64_t chunk_len = ((tiles + chunks - 1) / chunks) * 128;
    chunks = (shared_len + chunk_len - 1) / chunk_len;
    const int64_t Hkv = pool->num_kv_heads, d = pool->head_dim;
    const size_t need = cascade_bytes(batch, num_q_heads, Hkv, d, chunks);
    if (workspace_bytes < need)
        return fail(MINISGL_ERR_WORKSPACE, "cascade_decode_attn: workspace %zu bytes < %zu", workspace_bytes,
                    need);
    char *ws = static_cast<char *>(workspace);
    // prefix: chunk c is positions [c*chunk_len, ...) of the shared rows, read
    // from the first page-table row; every chunk reads q rows 0..B-1
    minisgl::ExtendArgs p;
    p.q = q;
    p.k_layer = layer_ptr(pool->k_base, pool, layer);
    p.v_layer = layer_ptr(pool->v_base, pool, layer);
    p.row_stride = pool->row_stride;
    p.num_rows = pool->num_rows;
    p.page_table = page_table;
    p.pt_stride = chunk_len;
    p.pt_width = (int32_t)chunk_len;
    p.cached_lens = p.extend_lens = p.q_offsets = nullptr;
    p.batch = (int32_t)chunks;
    p.total_q_tokens = (int32_t)(chunks * batch);
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = pool->num_kv_heads;
    p.head_dim = pool->head_dim;
    p.sm_scale = sm_scale;
    p.out = nullptr;
    p.prefix_only = 1;
    p.out_offsets = nullptr;
    p.prefix_chunk_len = (int32_t)chunk_len;
    p.prefix_len = shared_len;
    p.prefix_queries = batch;
    p.sched = reinterpret_cast<unsigned int *>(ws);
    ws += 256;
    const size_t vec = (size_t)batch * num_q_heads;
    minisgl::CascadeArgs c;
    c.pre_o = reinterpret_cast<float *>(ws);
    ws += align256((size_t)chunks * vec * d * 4);
    c.pre_lse = reinterpret_cast<float *>(ws);
    ws += align256((size_t)chunks * vec * 4);
    p.out_f32 = c.pre_o;
    p.lse_out = c.pre_lse;
    c.seq_lens = seq_lens;
    c.batch = batch;
    c.num_q_heads = num_q_heads;
    c.head_dim = pool->head_dim;
    c.shared_len = shared_len;
    c.chunks = (int32_t)chunks;
    c.out = out;
    minisgl::DecodeArgs &sd = c.suffix;  // the suffix: page table shifted by P columns
    sd.q = q;
    sd.k_layer = p.k_layer;
    sd.v_layer = p.v_layer;
    sd.row_stride = pool->row_stride;
    sd.num_rows = pool->num_rows;
    sd.page_table = page_table + shared_len;
    sd.pt_stride = pt_row_stride;
    sd.pt_width = pt_width - shared_len;
    sd.seq_lens = seq_lens;
    sd.len_offset = shared_len;
    sd.batch = batch;
    sd.num_q_heads = num_q_heads;
    sd.num_kv_heads = pool->num_kv_heads;
    sd.head_dim = pool->head_dim;
    sd.sm_scale = sm_scale;
    sd.out = nullptr;
    sd.split_count = reinterpret_cast<int32_t *>(ws);
    ws += align256((size_t)batch * Hkv * 4);
    sd.ws_lse = reinterpret_cast<float *>(ws);
    ws += align256(vec * CASCADE_SUFFIX_SPLITS * 4);
    sd.ws_o = reinterpret_cast<float *>(ws);
    sd.max_splits = CASCADE_SUFFIX_SPLITS;
    sd.split_tokens = 0;
    sd.lse_out = nullptr;
    sd.out_loc = nullptr;
    sd.k_new = sd.v_new = nullptr;
    sd.new_k_stride = sd.new_v_stride = 0;
    sd.partials_only = 1;
    return cuda_status(minisgl::launch_cascade(c, p, static_cast<cudaStream_t>(stream)),
                       "cascade_decode_attn");
}

size_t minisgl_cascade_extend_workspace_bytes(int32_t total_q_tokens, int32_t num_q_heads,
                                              int32_t head_dim) {
    if (total_q_tokens < 0 || num_q_heads < 1 || head_dim < 1) return 0;
    const size_t rows = (size_t)total_q_tokens * num_q_heads;
    return 256 + align256(rows * head_dim * 4) + align256(rows * 4);
}

int minisgl_cascade_extend_attn(const minisgl_kv_pool *pool, int32_t layer, const void *q,
                                int32_t num_q_heads, const int32_t *page_table, int32_t batch,
                                int64_t pt_row_stride, int32_t pt_width, const int32_t *cached_lens,
                                const int32_t *extend_lens, const int32_t *q_offsets,
                                int32_t total_q_tokens, int32_t shared_len, float sm_scale, void *out,
                                void *workspace, size_t workspace_bytes, void *stream) {
    g_err.clear();
    NvtxRange nvtx_range("minisgl_cascade_extend_attn");
    if (int rc = check_pool(pool, layer, "cascade_extend_attn")) return rc;
    if (int rc = check_heads(num_q_heads, pool->num_kv_heads, 16, "cascade_extend_attn")) return rc;
    if (batch < 0 || batch > 4096)
        return fail(MINISGL_ERR_ARG, "cascade_extend_attn: batch %d outside [0, 4096]", batch);
    if (total_q_tokens < 0) return fail(MINISGL_ERR_ARG, "cascade_extend_attn: total_q_tokens < 0");
    if (!(sm_scale > 0.f) || !(sm_scale < 3.0e38f))
        return fail(MINISGL_ERR_ARG, "cascade_extend_attn: sm_scale must be positive and finite");
    if (pt_width < 1 || pt_row_stride < pt_width)
        return fail(MINISGL_ERR_SHAPE, "cascade_extend_attn: need 1 <= pt_width <= pt_row_stride");
    if (shared_len < 1 || shared_len > pt_width)
        return fail(MINISGL_ERR_ARG, "cascade_extend_attn: shared_len %d outside [1, pt_width]", shared_len);
    if (batch == 0 || total_q_tokens == 0) return MINISGL_OK;
    if (!q || !page_table || !cached_lens || !extend_lens || !q_offsets || !out || !workspace)
        return fail(MINISGL_ERR_ARG, "cascade_extend_attn: NULL pointer argument");
    if (!aligned16(q) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(MINISGL_ERR_SHAPE, "cascade_extend_attn: q, out 16-byte and workspace 256-byte aligned");
    const size_t need = minisgl_cascade_extend_workspace_bytes(total_q_tokens, num_q_heads, pool->head_dim);
    if (workspace_bytes < need)
        return fail(MINISGL_ERR_WORKSPACE, "cascade_extend_attn: workspace %zu bytes < %zu", workspace_bytes,
                    need);
    char *ws = static_cast<char *>(workspace);
    const size_t rows = (size_t)total_q_tokens * num_q_heads;
    unsigned int *counter = reinterpret_cast<unsigned int *>(ws);
    float *pre_o = reinterpret_cast<float *>(ws + 256);
    float *pre_lse = reinterpret_cast<float *>(ws + 256 + align256(rows * pool->head_dim * 4));
    // the new tokens' common part: all of them against the P shared positions,
    // one pseudo-request whose page-table row is the first request's
    minisgl::ExtendArgs p;
    p.q = q;
    p.k_layer = layer_ptr(pool->k_base, pool, layer);
    p.v_layer = layer_ptr(pool->v_base, pool, layer);
    p.row_stride = pool->row_stride;
    p.num_rows = pool->num_rows;
    p.page_table = page_table;
    p.pt_stride = shared_len;
    p.pt_width = shared_len;
    p.cached_lens = p.extend_lens = p.q_offsets = nullptr;
    p.batch = 1;
    p.total_q_tokens = total_q_tokens;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = pool->num_kv_heads;
    p.head_dim = pool->head_dim;
    p.sm_scale = sm_scale;
    p.out = nullptr;
    p.prefix_only = 1;
    p.out_f32 = pre_o;
    p.lse_out = pre_lse;
    p.out_offsets = nullptr;
    p.prefix_chunk_len = shared_len;
    p.prefix_len = shared_len;
    p.prefix_queries = total_q_tokens;
    p.sched = counter;
    // each request's own positions, causally, with the common part folded in
    minisgl::ExtendArgs o = p;
    o.page_table = page_table + shared_len;
    o.pt_stride = pt_row_stride;
    o.pt_width = pt_width - shared_len;
    o.cached_lens = cached_lens;
    o.extend_lens = extend_lens;
    o.q_offsets = q_offsets;
    o.batch = batch;
    o.out = out;
    o.prefix_only = 0;
    o.out_f32 = nullptr;
    o.lse_out = nullptr;
    o.prefix_chunk_len = o.prefix_len = o.prefix_queries = 0;
    o.len_offset = shared_len;
    o.merge_o = pre_o;
    o.merge_lse = pre_lse;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (int rc = cuda_status(minisgl::launch_extend(p, st), "cascade_extend_attn")) return rc;
    return cuda_status(minisgl::launch_extend(o, st), "cascade_extend_attn");
}

int minisgl_rope_store_kv(const minisgl_kv_pool *pool, int32_t layer, void *q, int32_t num_q_heads,
                          int64_t q_tok_stride, const void *k, const void *v, int64_t k_tok_stride,
                          int64_t v_tok_stride, const int32_t *positions, const float *cos_sin_cache,
                          int32_t max_positions, const int32_t *out_loc, int32_t n_tokens,
                          void *stream) {
    g_err.clear();
    NvtxRange nvtx_range("minisgl_rope_store_kv");
    if (int rc = check_pool(pool, layer, "rope_store_kv")) return rc;
    if (num_q_heads < 1) return fail(MINISGL_ERR_ARG, "rope_store_kv: num_q_heads < 1");
    if (n_tokens < 0) return fail(MINISGL_ERR_ARG, "rope_store_kv: n_tokens < 0");
    if (max_positions < 1) return fail(MINISGL_ERR_ARG, "rope_store_kv: max_positions < 1");
    if (n_tokens == 0) return MINISGL_OK;
    if (!q || !k || !v || !positions || !cos_sin_cache || !out_loc)
        return fail(MINISGL_ERR_ARG, "rope_store_kv: NULL pointer argument");
    const int64_t d = pool->head_dim;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(cos_sin_cache))
        return fail(MINISGL_ERR_SHAPE, "rope_store_kv: q, k, v and the cos/sin table must be 16-byte aligned");
    if (q_tok_stride < (int64_t)num_q_heads * d || q_tok_stride % 8)
        return fail(MINISGL_ERR_SHAPE, "rope_store_kv: q token stride must be >= H_q*d and a multiple of 8");
    const int64_t row = (int64_t)pool->num_kv_heads * d;
    if (k_tok_stride < row || v_tok_stride < row || k_tok_stride % 8 || v_tok_stride % 8)
        return fail(MINISGL_ERR_SHAPE, "rope_store_kv: k/v token strides must be >= H_kv*d and multiples of 8");
    minisgl::RopeStoreArgs a;
    a.k_layer = const_cast<void *>(layer_ptr(pool->k_base, pool, layer));
    a.v_layer = const_cast<void *>(layer_ptr(pool->v_base, pool, layer));
    a.row_stride = pool->row_stride;
    a.num_rows = pool->num_rows;
    a.q = q;
    a.q_tok_stride = q_tok_stride;
    a.k = k;
    a.v = v;
    a.k_tok_stride = k_tok_stride;
    a.v_tok_stride = v_tok_stride;
    a.positions = positions;
    a.cos_sin = cos_sin_cache;
    a.max_positions = max_positions;
    a.out_loc = out_loc;
    a.n_tokens = n_tokens;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = pool->num_kv_heads;
    a.head_dim = (int32_t)d;
    return cuda_status(minisgl::launch_rope_store_kv(a, static_cast<cudaStream_t>(stream)),
                       "rope_store_kv");
}

int minisgl_check_indices(const int32_t *page_table, int32_t batch, int64_t pt_row_stride,
                          int32_t pt_width, const int32_t *lens, const int32_t *out_loc,
                          int32_t n_out, int32_t num_rows, uint32_t *counts, void *stream) {
    g_err.clear();
    NvtxRange nvtx_range("minisgl_check_indices");
    if (!counts) return fail(MINISGL_ERR_ARG, "check_indices: NULL counts");
    if (batch < 0 || n_out < 0 || pt_width < 0)
        return fail(MINISGL_ERR_ARG, "check_indices: negative batch, n_out or pt_width");
    if (num_rows < 1) return fail(MINISGL_ERR_ARG, "check_indices: num_rows must be positive");
    if (batch > 0 && (!page_table || !lens))
        return fail(MINISGL_ERR_ARG, "check_indices: NULL page_table or lens");
    if (n_out > 0 && !out_loc) return fail(MINISGL_ERR_ARG, "check_indices: NULL out_loc");
    if (batch > 0 && pt_row_stride < pt_width)
        return fail(MINISGL_ERR_SHAPE, "check_indices: need pt_width <= pt_row_stride");
    minisgl::CheckArgs a;
    a.page_table = page_table;
    a.pt_stride = pt_row_stride;
    a.pt_width = pt_width;
    a.batch = batch;
    a.lens = lens;
    a.out_loc = out_loc;
    a.n_out = n_out;
    a.num_rows = num_rows;
    a.counts = counts;
    return cuda_status(minisgl::launch_check_indices(a, static_cast<cudaStream_t>(stream)),
                       "check_indices");
}

int minisgl_check_shared_prefix(const int32_t *page_table, int32_t batch, int64_t pt_row_stride,
                                int32_t pt_width, int32_t shared_len, const int32_t *lens,
                                uint32_t *counts, void *stream) {
    g_err.clear();
    NvtxRange nvtx_range("minisgl_check_shared_prefix");
    if (!counts) return fail(MINISGL_ERR_ARG, "check_shared_prefix: NULL counts");
    if (batch < 0 || pt_width < 0)
        return fail(MINISGL_ERR_ARG, "check_shared_prefix: negative batch or pt_width");
    if (shared_len < 1 || shared_len > pt_width)
        return fail(MINISGL_ERR_ARG, "check_shared_prefix: shared_len %d outside [1, pt_width]", shared_len);
    if (batch > 0 && (!page_table || !lens))
        return fail(MINISGL_ERR_ARG, "check_shared_prefix: NULL page_table or lens");
    if (batch > 0 && pt_row_stride < pt_width)
        return fail(MINISGL_ERR_SHAPE, "check_shared_prefix: need pt_width <= pt_row_stride");
    return cuda_status(minisgl::launch_check_shared_prefix(page_table, batch, pt_row_stride, shared_len, lens,
                                                           counts, static_cast<cudaStream_t>(stream)),
                       "check_shared_prefix");
}

}  // extern "C"
