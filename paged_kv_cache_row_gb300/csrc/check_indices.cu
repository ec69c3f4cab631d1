// check_indices.cu -- count index values that would address rows outside the
// pool, on the device, without trapping.
//
// The attention and store kernels never check index values: page_table and
// out_loc live in device memory, and an entry outside [0, num_rows) is a
// caller error whose row the kernels clamp into the pool (results
// unspecified).  This kernel lets a caller find such entries in a debugging
// run: it reads exactly the entries a decode or extend call would read
// (page_table[r, j] for j < lens[r], out_loc[i] for i < n_out) and counts the
// bad ones, plus the lengths outside [0, pt_width].  The pages' page_table
// rows hold raw physical rows padded to a multiple of 32 (mini-sglang-learn,
// paged KV pool chapter, page_table alignment passage); past a request's
// length the entries are undefined and are not read.
#include "kernels.h"

namespace minisgl {

__global__ void __launch_bounds__(256) check_indices_kernel(CheckArgs a) {
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nth = (int64_t)gridDim.x * blockDim.x;
    unsigned bad_pt = 0, bad_loc = 0, bad_len = 0;
    const int64_t cells = (int64_t)a.batch * a.pt_width;
    for (int64_t k = tid; k < cells; k += nth) {
        const int r = (int)(k / a.pt_width), j = (int)(k - (int64_t)r * a.pt_width);
        const int n = min(max(__ldg(a.lens + r), 0), a.pt_width);
        if (j < n) {
            const int v = __ldg(a.page_table + (int64_t)r * a.pt_stride + j);
            bad_pt += (v < 0 || v >= a.num_rows) ? 1u : 0u;
        }
    }
    for (int64_t k = tid; k < a.n_out; k += nth) {
        const int v = __ldg(a.out_loc + k);
        bad_loc += (v < 0 || v >= a.num_rows) ? 1u : 0u;
    }
    for (int64_t k = tid; k < a.batch; k += nth) {
        const int n = __ldg(a.lens + k);
        bad_len += (n < 0 || n > a.pt_width) ? 1u : 0u;
    }
    // every lane of the warp gets here: one atomic per warp and counter
    bad_pt = __reduce_add_sync(0xffffffffu, bad_pt);
    bad_loc = __reduce_add_sync(0xffffffffu, bad_loc);
    bad_len = __reduce_add_sync(0xffffffffu, bad_len);
    if ((threadIdx.x & 31) == 0) {
        if (bad_pt) atomicAdd(a.counts + 0, bad_pt);
        if (bad_loc) atomicAdd(a.counts + 1, bad_loc);
        if (bad_len) atomicAdd(a.counts + 2, bad_len);
    }
}

cudaError_t launch_check_indices(const CheckArgs &a, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(a.counts, 0, 3 * sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    const int64_t work = max((int64_t)a.batch * a.pt_width, (int64_t)max(a.n_out, a.batch));
    if (work == 0) return cudaSuccess;
    int64_t grid = (work + 255) / 256;
    const int64_t cap = 4LL * max(device_sm_count(), 1);
    if (grid > cap) grid = cap;
    check_indices_kernel<<<(unsigned)grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

// The shared-prefix (cascade) calls trust their caller that the first
// shared_len page-table entries are the same rows in every request and that
// every request reads at least shared_len positions (mini-sglang-learn,
// radix-cache chapter: requests matching a cached prefix point at its rows).
// This kernel counts the entries that break the first condition
// (page_table[r, j] != page_table[0, j], j < shared_len) and the requests
// that break the second (lens[r] < shared_len).
__global__ void __launch_bounds__(256) check_shared_prefix_kernel(const int32_t *page_table, int batch,
                                                                  int64_t pt_stride, int shared_len,
                                                                  const int32_t *lens, uint32_t *counts) {
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nth = (int64_t)gridDim.x * blockDim.x;
    unsigned diff = 0, shorter = 0;
    const int64_t cells = (int64_t)batch * shared_len;
    for (int64_t k = tid; k < cells; k += nth) {
        const int r = (int)(k / shared_len), j = (int)(k - (int64_t)r * shared_len);
        if (r > 0) diff += __ldg(page_table + (int64_t)r * pt_stride + j) != __ldg(page_table + j) ? 1u : 0u;
    }
    for (int64_t k = tid; k < batch; k += nth) shorter += __ldg(lens + k) < shared_len ? 1u : 0u;
    diff = __reduce_add_sync(0xffffffffu, diff);
    shorter = __reduce_add_sync(0xffffffffu, shorter);
    if ((threadIdx.x & 31) == 0) {
        if (diff) atomicAdd(counts + 0, diff);
        if (shorter) atomicAdd(counts + 1, shorter);
    }
}

cudaError_t launch_check_shared_prefix(const int32_t *page_table, int32_t batch, int64_t pt_stride,
                                       int32_t shared_len, const int32_t *lens, uint32_t *counts,
                                       cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(counts, 0, 2 * sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    const int64_t work = max((int64_t)batch * shared_len, (int64_t)batch);
    if (work == 0) return cudaSuccess;
    int64_t grid = (work + 255) / 256;
    const int64_t cap = 4LL * max(device_sm_count(), 1);
    if (grid > cap) grid = cap;
    check_shared_prefix_kernel<<<(unsigned)grid, 256, 0, s>>>(page_table, batch, pt_stride, shared_len, lens,
                                                              counts);
    return cudaGetLastError();
}

}  // namespace minisgl
