"""The allocation-free decode entry point (minisgl_decode_attn_noalloc).

It exists for callers that cannot allocate device memory at run time -- an
engine that has given nearly all free HBM to its KV pool, code inside a host
application that owns the allocator, a decode loop that cannot afford
cudaMalloc/cudaFree -- and takes its split-KV scratch from a fixed array in the
library instead of a caller workspace.  These tests call it through the C ABI
(the ctypes binding) and check that it returns what the regular entry point
returns and what the fp64 oracle returns, on two calls in a row (the array
keeps the previous call's contents), that the largest batch whose scratch
fits is served, and that one request more is refused with a clear error.
The file is named to be collected last.
"""
import ctypes

import pytest
import torch

import oracle
import paged_kv_cache_row_gb300 as mk
import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
DEV = "cuda"
MAX_ABS, MEAN_ABS = gu.MAX_ABS, gu.MEAN_ABS  # the tolerance the other attention tests use
SCRATCH = 32 << 20  # bytes of the library's built-in array


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_row_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _case(seed, batch, lo, hi):
    return workloads.make_decode_case(f"noalloc-{seed}", num_layers=1, num_q_heads=16,
                                      num_kv_heads=8, head_dim=128, page_size=1, batch=batch,
                                      ctx_lo=lo, ctx_hi=hi, value_std=0.5, seed=seed)


def _run(case):
    """The no-alloc call against the workspace entry point and the oracle."""
    pool_t, k_new, v_new, q = workloads.make_decode_values(case, DEV)
    hk, hv = gu.u16(pool_t[0, 0]), gu.u16(pool_t[1, 0])
    pool = mk.KVPool(pool_t)
    pt, sl = case.page_table.to(DEV), case.seq_lens.to(DEV)
    mk.minisgl_store_kv(pool, 0, k_new[0], v_new[0], case.out_loc.to(DEV))
    ref = mk.minisgl_decode_attn(pool, 0, q[0], pt, sl, case.sm_scale)
    out = torch.full_like(ref, float("nan"))
    mk.minisgl_decode_attn_noalloc(pool, 0, q[0], pt, sl, case.sm_scale, out=out)
    torch.cuda.synchronize()
    err = (out.float() - ref.float()).abs()
    assert torch.isfinite(out.float()).all()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS, (case.name, err.max().item())
    orc = oracle.get()
    orc.store_kv(hk, hv, k_new[0].cpu(), v_new[0].cpu(), case.out_loc)
    exp, _ = gu.parallel_oracle_decode(hk, hv, q[0], case.page_table, case.seq_lens, case.sm_scale)
    gu.check_attn(out, exp, f"{case.name} no-alloc vs oracle")


def test_noalloc_matches_workspace_entry_point_and_oracle_twice():
    # two calls in a row on different batches: the second finds the first's
    # leftovers in the shared scratch array and must not be affected by them
    for seed, batch, lo, hi in [(501, 64, 512, 4096), (502, 9, 1, 700)]:
        _run(_case(seed, batch, lo, hi))


def _largest_batch_that_fits(hq=16, hkv=8, d=128):
    b = 1
    while mk.minisgl_decode_workspace_bytes(b + 1, hq, hkv, d, 2) <= SCRATCH:
        b += 1
    return b


def test_noalloc_serves_the_largest_batch_that_fits():
    b = _largest_batch_that_fits()
    assert b == 2028  # the figure the header documents for 16 query / 8 KV heads at d 128
    _run(_case(503, b, 1, 40))


def test_noalloc_rejects_sizes_beyond_the_array():
    lib = mk.load_library()
    fake = 1 << 40  # never dereferenced: the size check comes first
    d = mk._PoolDesc(k_base=fake, v_base=fake, layer_stride=8 * 128 * 1000, row_stride=8 * 128,
                     num_layers=1, num_rows=1000, num_kv_heads=8, head_dim=128, page_size=1,
                     dtype=mk.MINISGL_BF16)
    for batch, hq in [(_largest_batch_that_fits() + 1, 16), (4096, 128)]:
        rc = lib.minisgl_decode_attn_noalloc(ctypes.byref(d), 0, fake, hq, fake, batch, 32, 32, fake,
                                             0.1, fake, 0, None)
        assert rc == -6  # MINISGL_ERR_WORKSPACE
        assert b"built-in" in lib.minisgl_last_error()
