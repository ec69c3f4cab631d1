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

}  // namespace minisgl
