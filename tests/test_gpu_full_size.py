"""Full-size parity for the five workloads, in the launch configuration the
benchmark times: every layer of the step is run, and EVERY output element of
the checked layers (all requests, padding requests included, all heads; every
new token of every extend batch) is compared with the fp64 oracle, which runs
on one thread per host core.  The pool after the step is compared with the
oracle's store_kv byte for byte.
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


def run_decode_full(case, check_layers, fused=False):
    """One decode step over all layers (store_kv + decode per layer, or the
    fused call), then every output of `check_layers` against the oracle."""
    pool_t, k_new, v_new, q = workloads.make_decode_values(case, DEV)
    pool = mk.KVPool(pool_t, case.page_size)
    pt, sl, loc = case.page_table.to(DEV), case.seq_lens.to(DEV), case.out_loc.to(DEV)
    # oracle inputs: the whole layer as the generator drew it, before any kernel runs
    snaps = {l: (gu.u16(pool_t[0, l]), gu.u16(pool_t[1, l])) for l in check_layers}
    ws = mk.decode_workspace(case.batch, case.num_q_heads, pool)
    outs = {}
    for l in range(case.num_layers):  # the whole step, as the benchmark runs it
        if fused:
            o = mk.minisgl_store_decode_attn(pool, l, k_new[l], v_new[l], loc, q[l], pt, sl,
                                             case.sm_scale, workspace=ws)
        else:
            mk.minisgl_store_kv(pool, l, k_new[l], v_new[l], loc)
            o = mk.minisgl_decode_attn(pool, l, q[l], pt, sl, case.sm_scale, workspace=ws)
        if l in check_layers:
            outs[l] = o.clone()
    torch.cuda.synchronize()
    orc = oracle.get()
    for l in check_layers:
        hk, hv = snaps[l]
        orc.store_kv(hk, hv, k_new[l].cpu(), v_new[l].cpu(), case.out_loc)
        assert np.array_equal(gu.u16(pool_t[0, l]), hk), f"layer {l}: K pool differs from oracle store_kv"
        assert np.array_equal(gu.u16(pool_t[1, l]), hv), f"layer {l}: V pool differs from oracle store_kv"
        ref, _ = gu.parallel_oracle_decode(hk, hv, q[l], case.page_table, case.seq_lens, case.sm_scale)
        stats = gu.check_attn(outs[l], ref, f"{case.name} layer {l} (all {case.batch} requests)")
        print(f"{case.name} layer {l}: {stats}")
    return pool_t, k_new, v_new, outs


def test_full_tiny_decode():
    case = workloads.decode_tiny()
    run_decode_full(case, [0])


@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused_store"])
def test_full_qwen3_0p6b_decode(fused):
    case = workloads.decode_qwen3_0p6b()
    run_decode_full(case, [0, case.num_layers - 1], fused=fused)


@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused_store"])
def test_full_llama3_8b_decode_with_padding(fused):
    """The headline workload: 32 layers, 200 real + 56 padding requests."""
    case = workloads.decode_llama3_8b()
    pool_t, k_new, v_new, outs = run_decode_full(case, [0, case.num_layers - 1], fused=fused)
    D = case.dummy_row
    G = case.num_q_heads // case.num_kv_heads
    for l, o in outs.items():
        # every padding request reads only the dummy row, whose V is the padding value
        vd = v_new[l][case.num_real]            # [H_kv, d]
        assert torch.equal(pool_t[1, l, D], vd)
        exp = vd.repeat_interleave(G, dim=0)    # [H_q, d]
        for r in range(case.num_real, case.batch):
            assert torch.equal(o[r], exp), "padding request output != V[dummy]"


def test_full_long_page64_decode():
    case = workloads.decode_long_page64()
    run_decode_full(case, [0])
    run_decode_full(case, [0], fused=True)


def test_full_radix_shared_extend():
    """Every new token of every chunked-prefill batch against the oracle, for
    the extend call and for the shared-prefix (cascade) extend call."""
    case = workloads.extend_radix_shared()
    assert 2 <= len(case.batches) <= 5
    pool_t, per_batch = workloads.make_extend_values(case, DEV)
    hk, hv = gu.u16(pool_t[0, 0]), gu.u16(pool_t[1, 0])  # ~0.2 GB: the whole pool
    pool = mk.KVPool(pool_t)
    orc = oracle.get()
    for bi, (b, (k, v, q)) in enumerate(zip(case.batches, per_batch)):
        assert b.total_tokens <= 8192
        mk.minisgl_store_kv(pool, 0, k, v, b.out_loc.to(DEV))
        o = mk.minisgl_extend_attn(pool, 0, q, b.page_table.to(DEV), b.cached_lens.to(DEV),
                                   b.extend_lens.to(DEV), b.q_offsets.to(DEV), case.sm_scale)
        torch.cuda.synchronize()
        orc.store_kv(hk, hv, k.cpu(), v.cpu(), b.out_loc)
        assert np.array_equal(gu.u16(pool_t[0, 0]), hk), f"batch {bi}: K pool differs"
        assert np.array_equal(gu.u16(pool_t[1, 0]), hv), f"batch {bi}: V pool differs"
        ref = gu.parallel_oracle_extend(hk, hv, q, b.page_table, b.cached_lens, b.extend_lens,
                                        b.q_offsets, case.sm_scale)
        stats = gu.check_attn(o, ref, f"extend batch {bi} (all {b.total_tokens} tokens)")
        print(f"extend batch {bi}: {stats}")
        # the shared-prefix (cascade) extend of the same batch: same oracle values
        oc = mk.minisgl_cascade_extend_attn(pool, 0, q, b.page_table.to(DEV), b.cached_lens.to(DEV),
                                            b.extend_lens.to(DEV), b.q_offsets.to(DEV),
                                            int(case.prefix_rows.numel()), case.sm_scale)
        torch.cuda.synchronize()
        stats = gu.check_attn(oc, ref, f"cascade extend batch {bi} (all {b.total_tokens} tokens)")
        print(f"cascade extend batch {bi}: {stats}")
    assert mk.minisgl_debug_timeout_count() == 0


def test_extend_long_context_full_budget():
    """One launch at the chunk budget: a request extending 2,000 tokens over
    24,000 cached ones beside a 6,192-token prefill with nothing cached (8,192
    new tokens in all, GQA 4).  Sampled rows are checked against the oracle as
    decodes over positions 0 .. C + t."""
    cached, ext = [24000, 0], [2000, 6192]
    Hq, Hkv = 32, 8
    g = torch.Generator().manual_seed(2024)
    lens = [c + e for c, e in zip(cached, ext)]
    R = sum(lens) + 64
    perm = torch.randperm(R - 1, generator=g).to(torch.int32)
    W = workloads.align_up(max(lens))
    pt = torch.full((2, W), R - 1, dtype=torch.int32)
    locs, off = [], 0
    for r, n in enumerate(lens):
        pt[r, :n] = perm[off:off + n]
        locs.append(perm[off + cached[r]:off + n])
        off += n
    case = workloads.ExtendCase(name="long-extend", num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128,
                                num_rows=R, prefix_rows=perm[:0], extend_lens=list(ext),
                                sm_scale=1 / 128 ** 0.5, value_std=0.5, seed=2024)
    b = workloads.ExtendBatch(req_ids=[0, 1], cached_lens=torch.tensor(cached, dtype=torch.int32),
                              extend_lens=torch.tensor(ext, dtype=torch.int32),
                              q_offsets=torch.tensor([0, ext[0], ext[0] + ext[1]], dtype=torch.int32),
                              page_table=pt, out_loc=torch.cat(locs).to(torch.int32))
    case.batches.append(b)
    assert b.total_tokens == 8192
    pool_t, per_batch = workloads.make_extend_values(case, DEV)
    host = (gu.u16(pool_t[0, 0]), gu.u16(pool_t[1, 0]))
    k, v, q = per_batch[0]
    pool = mk.KVPool(pool_t)
    mk.minisgl_store_kv(pool, 0, k, v, b.out_loc.to(DEV))
    o = mk.minisgl_extend_attn(pool, 0, q, b.page_table.to(DEV), b.cached_lens.to(DEV),
                               b.extend_lens.to(DEV), b.q_offsets.to(DEV), case.sm_scale)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()
    orc = oracle.get()
    orc.store_kv(host[0], host[1], k.cpu(), v.cpu(), b.out_loc)
    gen = torch.Generator().manual_seed(5)
    for r in range(2):
        C, E, a0 = cached[r], ext[r], int(b.q_offsets[r])
        ts = sorted({0, 1, 127, 128, E - 1, E // 2} | set(torch.randint(0, E, (6,), generator=gen).tolist()))
        qs = q[[a0 + t for t in ts]].cpu()
        sl = torch.tensor([C + t + 1 for t in ts], dtype=torch.int32)
        ref, _ = orc.decode(qs, host[0], host[1], pt[r:r + 1].repeat(len(ts), 1), sl, case.sm_scale)
        gu.check_attn(o[[a0 + t for t in ts]], ref, f"long extend request {r}")
    assert mk.minisgl_debug_timeout_count() == 0
