"""GPU parity of the fused RoPE + store_kv call against the fp64 oracle.

The rotated q (in place) and the rotated k written into the pool are compared
element by element with oracle_rope: the kernel computes in fp32 and rounds
to bf16, so each value must lie within half a bf16 ulp of the exact result
(at most 2^-8 of its magnitude) plus the fp32 rounding of the products,
bounded by 2^-20 (|x1| + |x2|).  v rows must be
bit-exact (oracle store_kv), rows outside out_loc untouched, and the k input
unchanged.  All calls go through the C ABI (the ctypes binding).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_row_gb300 as mk
import workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_row_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def rope_bound(x: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Allowed |gpu - exact| per element: half a bf16 ulp of the result (at
    most 2^-8 |result|) plus the fp32 error of x1*c - x2*s (below 2^-20 (|x1| + |x2|))."""
    d = x.shape[-1]
    h = d // 2
    pair = np.abs(x[..., :h]) + np.abs(x[..., h:])
    pair = np.concatenate([pair, pair], -1)
    return 2.0 ** -8 * np.abs(ref) + 2.0 ** -20 * pair + 1e-30


def check_rope(gpu: torch.Tensor, x_in: torch.Tensor, ref: np.ndarray, what: str):
    g = gpu.detach().float().cpu().double().numpy()
    x = x_in.detach().float().cpu().double().numpy()
    assert g.shape == ref.shape
    err = np.abs(g - ref)
    bad = err > rope_bound(x, ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off, max err {err.max():.3g}"


def run_rope(Hq, Hkv, d, positions, out_loc, R, seed, max_pos, dummy_from=None, layers=1, layer=0,
             pagefirst=False):
    g = torch.Generator(device=DEV).manual_seed(seed)
    N = out_loc.numel()
    if pagefirst:  # rows outermost in memory, seen as the logical (2, L, R, H_kv, d) view
        base = torch.empty((2, R, layers, Hkv, d), dtype=torch.bfloat16, device=DEV).normal_(0, 0.5, generator=g)
        pool_t = base.permute(0, 2, 1, 3, 4)
    else:
        pool_t = torch.empty((2, layers, R, Hkv, d), dtype=torch.bfloat16, device=DEV).normal_(0, 0.5, generator=g)
    q = torch.empty((N, Hq, d), dtype=torch.bfloat16, device=DEV).normal_(0, 0.5, generator=g)
    k = torch.empty((N, Hkv, d), dtype=torch.bfloat16, device=DEV).normal_(0, 0.5, generator=g)
    v = torch.empty((N, Hkv, d), dtype=torch.bfloat16, device=DEV).normal_(0, 0.5, generator=g)
    if dummy_from is not None:  # padding tokens: identical k, v (and positions)
        k[dummy_from:] = k[dummy_from:dummy_from + 1].clone()
        v[dummy_from:] = v[dummy_from:dummy_from + 1].clone()
    table = workloads.rope_cos_sin_cache(d, max_pos).to(DEV)
    q_in, k_in = q.clone(), k.clone()
    hk, hv = gu.u16(pool_t[0, layer]), gu.u16(pool_t[1, layer])
    other = [gu.u16(pool_t[kv, l]) for kv in (0, 1) for l in range(layers) if l != layer]
    pool = mk.KVPool(pool_t)
    mk.minisgl_rope_store_kv(pool, layer, q, k, v, positions.to(DEV), table, out_loc.to(DEV))
    torch.cuda.synchronize()
    orc = oracle.get()
    tab = table.cpu()
    ref_q = orc.rope(q_in.cpu(), positions, tab)
    ref_k = orc.rope(k_in.cpu(), positions, tab)
    check_rope(q, q_in, ref_q, "q")
    assert torch.equal(k, k_in), "k input must stay unrotated"
    # v and untouched rows through the oracle's store_kv (k rows written below)
    orc.store_kv(hk, hv, k_in.cpu(), v.cpu(), out_loc)
    gk, gv = gu.u16(pool_t[0, layer]), gu.u16(pool_t[1, layer])
    assert np.array_equal(gv, hv), "V pool differs from oracle store_kv"
    rows = torch.unique(out_loc.to(torch.int64))
    mask = np.ones(R, dtype=bool)
    mask[rows.numpy()] = False
    assert np.array_equal(gk[mask], hk[mask]), "a K row outside out_loc changed"
    # each written K row holds the rotated k of (one of) its tokens
    last = {}
    for i, r in enumerate(out_loc.tolist()):
        last[r] = i
    idx = torch.tensor([last[int(r)] for r in rows.tolist()])
    kd = pool_t[0, layer, rows.to(DEV)]
    check_rope(kd, k_in[idx.to(DEV)], ref_k[idx.numpy()], "pool K rows")
    for j, l in enumerate(l for l in range(layers) if l != layer):
        assert np.array_equal(gu.u16(pool_t[0, l]), other[j]), "another layer's K changed"
        assert np.array_equal(gu.u16(pool_t[1, l]), other[len(other) // 2 + j]), "another layer's V changed"
    return q, pool_t


SMALL = [
    # Hq, Hkv, d, N, R, max_pos
    (8, 2, 64, 37, 100, 300),
    (16, 8, 128, 129, 400, 5000),
    (32, 8, 128, 300, 700, 9000),
    (4, 4, 128, 1, 20, 10),
    (64, 8, 128, 70, 200, 33000),
]


@pytest.mark.parametrize("Hq,Hkv,d,N,R,max_pos", SMALL)
def test_rope_store_kv_small(Hq, Hkv, d, N, R, max_pos):
    g = torch.Generator().manual_seed(N * 7 + d)
    positions = torch.randint(0, max_pos, (N,), generator=g).to(torch.int32)
    positions[0] = max_pos - 1  # last table row
    out_loc = torch.randperm(R, generator=g)[:N].to(torch.int32)
    run_rope(Hq, Hkv, d, positions, out_loc, R, seed=N, max_pos=max_pos, layers=2, layer=1)


def test_rope_store_kv_padding_requests_share_the_dummy_row():
    # 20 real tokens at fresh rows, 12 padding tokens all writing the dummy row
    R, n_real, n_pad = 64, 20, 12
    g = torch.Generator().manual_seed(5)
    out_loc = torch.cat([torch.randperm(R - 2, generator=g)[:n_real],
                         torch.full((n_pad,), R - 2)]).to(torch.int32)
    positions = torch.cat([torch.randint(1, 500, (n_real,), generator=g),
                           torch.zeros(n_pad, dtype=torch.int64)]).to(torch.int32)
    run_rope(16, 4, 128, positions, out_loc, R, seed=6, max_pos=512, dummy_from=n_real)


def test_rope_store_kv_empty_is_noop():
    pool_t = torch.zeros((2, 1, 8, 2, 64), dtype=torch.bfloat16, device=DEV)
    q = torch.zeros((0, 4, 64), dtype=torch.bfloat16, device=DEV)
    kv = torch.zeros((0, 2, 64), dtype=torch.bfloat16, device=DEV)
    e = torch.zeros(0, dtype=torch.int32, device=DEV)
    mk.minisgl_rope_store_kv(mk.KVPool(pool_t), 0, q, kv, kv,
                             e, workloads.rope_cos_sin_cache(64, 4).to(DEV), e)
    torch.cuda.synchronize()
    assert not bool(pool_t.any())


def test_rope_store_kv_extend_batch_full_size():
    """The first radix-shared chunked-prefill batch (8192 tokens, H_q 32, H_kv 8)."""
    case = workloads.extend_radix_shared()
    b = case.batches[0]
    pos = workloads.extend_positions(b)
    run_rope(case.num_q_heads, case.num_kv_heads, case.head_dim, pos, b.out_loc, case.num_rows,
             seed=11, max_pos=int(pos.max()) + 1)


def test_rope_then_decode_matches_oracle():
    """The fused call feeding decode attention: rope_store_kv of the step's
    tokens, then decode over the pool; the oracle rotates, stores and attends
    on its own copy."""
    case = workloads.decode_tiny()
    pool_t, k_new, v_new, q = workloads.make_decode_values(case, DEV)
    hk, hv = gu.u16(pool_t[0, 0]), gu.u16(pool_t[1, 0])
    pos = workloads.decode_positions(case)
    table = workloads.rope_cos_sin_cache(case.head_dim, int(pos.max()) + 1).to(DEV)
    q0, k0, v0 = q[0].clone(), k_new[0].clone(), v_new[0].clone()
    pool = mk.KVPool(pool_t)
    mk.minisgl_rope_store_kv(pool, 0, q[0], k_new[0], v_new[0], pos.to(DEV), table,
                             case.out_loc.to(DEV))
    out = mk.minisgl_decode_attn(pool, 0, q[0], case.page_table.to(DEV), case.seq_lens.to(DEV),
                                 case.sm_scale)
    torch.cuda.synchronize()
    orc = oracle.get()
    tab = table.cpu()
    # the oracle's rotated values are rounded to bf16 the way the kernel stores them
    rq = torch.from_numpy(orc.rope(q0.cpu(), pos, tab)).to(torch.bfloat16)
    rk = torch.from_numpy(orc.rope(k0.cpu(), pos, tab)).to(torch.bfloat16)
    orc.store_kv(hk, hv, rk, v0.cpu(), case.out_loc)
    ref, _ = orc.decode(rq, hk, hv, case.page_table, case.seq_lens, case.sm_scale)
    gu.check_attn(out, ref, "rope -> store -> decode")


def test_rope_store_kv_pagefirst_pool():
    """RoPE + store_kv into layer 2 of a PageFirst pool (row stride 3*H_kv*d):
    the rotated k rows land in that layer only."""
    g = torch.Generator().manual_seed(61)
    N, R, max_pos = 90, 300, 4000
    pos = torch.randint(0, max_pos, (N,), generator=g).to(torch.int32)
    loc = torch.randperm(R, generator=g)[:N].to(torch.int32)
    run_rope(16, 4, 128, pos, loc, R, 62, max_pos, layers=3, layer=2, pagefirst=True)
