"""GPU parity of the shared-prefix (cascade) decode call against the fp64 oracle.

The oracle is plain decode over each request's full page-table row: cascade
decode must compute exactly that, only reading the shared rows once.  Cases
span group sizes 1-16, prefixes shorter than one tile, ending on and off tile
edges, batches wider than one query block, empty private suffixes and the
full 64-request, 4096-token-prefix workload of the benchmark.  All calls go
through the C ABI (the ctypes binding).
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


def run_cascade(case, shared_len, seq_override=None, pagefirst=False):
    pool_t, k_new, v_new, q = workloads.make_decode_values(case, DEV)
    hk, hv = gu.u16(pool_t[0, 0]), gu.u16(pool_t[1, 0])
    layer = 0
    if pagefirst:  # the same rows as layer 1 of a 2-layer PageFirst pool
        _, _, R, Hkv, d = pool_t.shape
        g = torch.Generator(device=DEV).manual_seed(case.seed + 1)
        base = torch.empty((2, R, 2, Hkv, d), dtype=torch.bfloat16, device=DEV).normal_(0, 0.5, generator=g)
        view = base.permute(0, 2, 1, 3, 4)
        view[:, 1] = pool_t[:, 0]
        pool_t, layer = view, 1
    pool = mk.KVPool(pool_t)
    seq = case.seq_lens.clone() if seq_override is None else seq_override
    pt, sl, loc = case.page_table.to(DEV), seq.to(DEV), case.out_loc.to(DEV)
    mk.minisgl_store_kv(pool, layer, k_new[0], v_new[0], loc)
    out = mk.minisgl_cascade_decode_attn(pool, layer, q[0], pt, sl, shared_len, case.sm_scale)
    plain = mk.minisgl_decode_attn(pool, layer, q[0], pt, sl, case.sm_scale)
    torch.cuda.synchronize()
    orc = oracle.get()
    orc.store_kv(hk, hv, k_new[0].cpu(), v_new[0].cpu(), case.out_loc)
    ref, _ = gu.parallel_oracle_decode(hk, hv, q[0], case.page_table, seq, case.sm_scale)
    gu.check_attn(out, ref, f"{case.name} cascade")
    gu.check_attn(plain, ref, f"{case.name} plain decode")
    assert mk.minisgl_debug_timeout_count() == 0, "a tensor-core kernel wait ran out"
    return out


CASES = [
    # Hq, Hkv, B, prefix, suffix_lo, suffix_hi
    (8, 2, 5, 70, 0, 40),
    (32, 8, 200, 300, 1, 700),
    (64, 8, 9, 129, 0, 3),
    (4, 4, 3, 128, 5, 5),
    (32, 2, 7, 1, 1, 300),
    (16, 8, 33, 1000, 0, 200),
]


@pytest.mark.parametrize("Hq,Hkv,B,P,lo,hi", CASES)
def test_cascade_decode_small(Hq, Hkv, B, P, lo, hi):
    case = workloads.make_shared_prefix_decode_case(f"cascade-g{Hq // Hkv}-p{P}", num_q_heads=Hq,
                                                    num_kv_heads=Hkv, head_dim=128, batch=B,
                                                    prefix_len=P, suffix_lo=lo, suffix_hi=hi,
                                                    seed=B * 31 + P)
    run_cascade(case, P)


@pytest.mark.parametrize("Hq,Hkv,d", [(6, 2, 128), (10, 2, 64), (12, 2, 64), (14, 2, 128), (8, 8, 64)])
def test_cascade_decode_head_dims_and_odd_groups(Hq, Hkv, d):
    """head_dim 64 and group sizes that do not divide the 128-row tile."""
    case = workloads.make_shared_prefix_decode_case(f"cascade-g{Hq // Hkv}-d{d}", num_q_heads=Hq,
                                                    num_kv_heads=Hkv, head_dim=d, batch=37,
                                                    prefix_len=700, suffix_lo=0, suffix_hi=300,
                                                    seed=Hq * 7 + d)
    run_cascade(case, 700)


def test_cascade_decode_prefix_fills_the_gpu():
    """A batch whose prefix part keeps every SM busy (64 query heads, 200
    requests, 4096 shared positions): the two parts run one after the other
    on the caller's stream instead of side by side."""
    case = workloads.make_shared_prefix_decode_case("cascade-wide", num_q_heads=64, num_kv_heads=8,
                                                    head_dim=128, batch=200, prefix_len=4096,
                                                    suffix_lo=0, suffix_hi=100, seed=97)
    run_cascade(case, 4096)


def test_cascade_decode_two_calls_in_a_row_on_side_streams():
    """Consecutive cascade calls on two caller streams share the library's
    second stream; both results stay exact."""
    c1 = workloads.decode_shared_prefix_qwen3(prefix_len=1024)
    c2 = workloads.make_shared_prefix_decode_case("cascade-second", num_q_heads=16, num_kv_heads=8,
                                                  head_dim=128, batch=48, prefix_len=2000,
                                                  suffix_lo=0, suffix_hi=400, seed=98)
    orc = oracle.get()
    runs = []
    for case in (c1, c2):
        pool_t, k_new, v_new, q = workloads.make_decode_values(case, DEV)
        hk, hv = gu.u16(pool_t[0, 0]), gu.u16(pool_t[1, 0])
        pool = mk.KVPool(pool_t)
        pt, sl = case.page_table.to(DEV), case.seq_lens.to(DEV)
        mk.minisgl_store_kv(pool, 0, k_new[0], v_new[0], case.out_loc.to(DEV))
        orc.store_kv(hk, hv, k_new[0].cpu(), v_new[0].cpu(), case.out_loc)
        ws = torch.zeros(mk.minisgl_cascade_workspace_bytes(case.batch, case.num_q_heads,
                                                            case.num_kv_heads, case.head_dim),
                         dtype=torch.uint8, device=DEV)
        runs.append((case, pool, q[0], pt, sl, torch.empty_like(q[0]), ws, (hk, hv)))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for _ in range(3):
        for (case, pool, q, pt, sl, out, ws, _), st in zip(runs, streams):
            with torch.cuda.stream(st):
                mk.minisgl_cascade_decode_attn(pool, 0, q, pt, sl, case.shared_len, case.sm_scale,
                                               out=out, workspace=ws)
    torch.cuda.synchronize()
    for case, pool, q, pt, sl, out, ws, (hk, hv) in runs:
        ref, _ = gu.parallel_oracle_decode(hk, hv, q, case.page_table, case.seq_lens, case.sm_scale)
        gu.check_attn(out, ref, f"{case.name} on a side stream")
    assert mk.minisgl_debug_timeout_count() == 0


def test_cascade_decode_empty_suffixes():
    """Requests whose whole context is the shared prefix (no private rows):
    only the prefix contributes."""
    case = workloads.make_shared_prefix_decode_case("cascade-empty", num_q_heads=16, num_kv_heads=4,
                                                    head_dim=128, batch=6, prefix_len=200,
                                                    suffix_lo=0, suffix_hi=30, seed=3)
    seq = case.seq_lens.clone()
    seq[0] = 200
    seq[3] = 200
    run_cascade(case, 200, seq_override=seq)


def test_cascade_decode_shared_len_shorter_than_sharing():
    """Declaring fewer shared positions than the rows actually shared is
    still exact (the rest is treated as private)."""
    case = workloads.make_shared_prefix_decode_case("cascade-short", num_q_heads=8, num_kv_heads=8,
                                                    head_dim=128, batch=4, prefix_len=400,
                                                    suffix_lo=3, suffix_hi=90, seed=4)
    run_cascade(case, 137)


def test_cascade_decode_full_workload():
    run_cascade(workloads.decode_shared_prefix_qwen3(), 4096)


def test_cascade_decode_pagefirst_pool():
    """Cascade decode on layer 1 of a PageFirst pool (row stride 2*H_kv*d)."""
    case = workloads.make_shared_prefix_decode_case("cascade-pagefirst", num_q_heads=16, num_kv_heads=4,
                                                    head_dim=128, batch=12, prefix_len=400,
                                                    suffix_lo=0, suffix_hi=150, seed=71)
    run_cascade(case, 400, pagefirst=True)


def test_cascade_decode_large_batch():
    """1024 requests sharing a 600-token prefix, GQA 4: many prefix query
    blocks per KV head and many suffix streams."""
    case = workloads.make_shared_prefix_decode_case("cascade-b1024", num_q_heads=16, num_kv_heads=4,
                                                    head_dim=128, batch=1024, prefix_len=600,
                                                    suffix_lo=0, suffix_hi=120, seed=1024)
    run_cascade(case, 600)


def test_cascade_decode_whole_table_shared():
    """shared_len equal to the page-table width and every request reading
    exactly the shared prefix: the suffix part has no columns at all."""
    case = workloads.make_shared_prefix_decode_case("cascade-all-shared", num_q_heads=16, num_kv_heads=8,
                                                    head_dim=128, batch=10, prefix_len=256,
                                                    suffix_lo=0, suffix_hi=0, seed=6)
    P = 256
    case.page_table = case.page_table[:, :P].contiguous()  # width 256, a multiple of 32
    seq = torch.full((case.batch,), P, dtype=torch.int32)
    run_cascade(case, P, seq_override=seq)
