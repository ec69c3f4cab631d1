// decode_noalloc.cu -- decode attention for callers that cannot allocate
// device memory.
//
// minisgl_decode_attn needs a scratch workspace for its split-KV partial
// results, and leaves it to the caller to provide one.  Some callers cannot:
// a serving engine that has already handed nearly all free HBM to its KV
// pool has nothing left to allocate from at run time; code embedded in a
// host application that owns the device allocator may have no way to ask it
// for memory; and a latency-critical decode loop cannot afford cudaMalloc /
// cudaFree, which may synchronise the device.  For them this file provides
// minisgl_decode_attn_noalloc, which runs the same kernels with the scratch
// taken from a fixed array that lives in the library's own device memory.
//
// The array (kNoallocScratchBytes = 32 MiB) is a file-scope static __device__
// variable: every GPU on which the library is loaded holds one copy of it
// until the process exits.  Host code cannot use the array's name as a device
// address -- on the host it names a stand-in object -- so every call, with
// its device current, looks the address up with cudaGetSymbolAddress (a
// host-side lookup) and checks the result.  Nothing is cached: if the caller
// resets the device and the module is loaded again, the array may sit at a
// new address, and a cached one would point at freed memory.  The first call
// on a device also loads the library's module there, so make that first call
// before any stream capture.  No call allocates or frees anything.
//
// Every call shares the one array and it keeps whatever the previous call
// left in it.  Nothing in it has to start at zero: the partial kernel writes
// every split count, partial output and LSE that the merge kernel later reads
// in the same call.  Two calls whose kernels overlap on the GPU (for example
// on two streams without ordering between them) race on the array and give
// wrong results; callers must order such calls.
#include <cstdio>

#include "kernels.h"
#include "minisgl.h"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of the scratch array on the current device, looked up on
// every call (see above for why it is not cached).
cudaError_t scratch_address(void **out) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" int minisgl_decode_attn_noalloc(const minisgl_kv_pool *pool, int32_t layer,
                                           const void *q, int32_t num_q_heads,
                                           const int32_t *page_table, int32_t batch,
                                           int64_t pt_row_stride, int32_t pt_width,
                                           const int32_t *seq_lens, float sm_scale, void *out,
                                           int32_t split_tokens, void *stream) {
    if (batch > 0 && pool && pool->num_kv_heads > 0 && num_q_heads > 0) {
        const size_t need = minisgl_decode_workspace_bytes(batch, num_q_heads, pool->num_kv_heads,
                                                           pool->head_dim, 2);
        if (need > kNoallocScratchBytes) {
            char msg[256];
            snprintf(msg, sizeof msg,
                     "decode_attn_noalloc: batch %d with %d query heads of dim %d needs %zu bytes of "
                     "scratch, more than the built-in %zu; use minisgl_decode_attn with a workspace",
                     batch, num_q_heads, pool->head_dim, need, kNoallocScratchBytes);
            return minisgl::report_error(MINISGL_ERR_WORKSPACE, msg);
        }
    }
    void *scratch = nullptr;
    if (batch > 0) {
        const cudaError_t e = scratch_address(&scratch);
        if (e != cudaSuccess) {
            char msg[256];
            snprintf(msg, sizeof msg, "decode_attn_noalloc: cudaGetSymbolAddress failed: %s",
                     cudaGetErrorString(e));
            return minisgl::report_error(MINISGL_ERR_CUDA, msg);
        }
    }
    // the regular entry point does every other check and the launches
    return minisgl_decode_attn(pool, layer, q, num_q_heads, page_table, batch, pt_row_stride,
                               pt_width, seq_lens, sm_scale, out, scratch, kNoallocScratchBytes,
                               split_tokens, stream);
}
