"""CUDA-Graph capture and replay of the decode and extend calls.

A serving engine replays the decode step as a CUDA graph with fixed buffers
(sglang-kernel guide, CUDA Graph passage: decode batches are padded to a
captured size and replayed), so every call must be capturable: no host
synchronisation, no allocation, no host-side branching on device data.  Each
test runs the calls eagerly, captures the same calls into a graph, replays the
graph twice and requires the replayed outputs to equal the eager ones bit for
bit (the kernels are deterministic for fixed inputs), and the eager outputs to
match the oracle.
"""
import zlib

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


def _capture(fn):
    """Warm up `fn` on a side stream, capture it, and return the graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("split_tokens", [0, 32])
def test_graph_store_decode_layers(split_tokens):
    """Three layers of fused store + decode per replay (padding requests
    included, as a padded CUDA-graph batch has them)."""
    name = f"graph-decode-{split_tokens}"
    case = workloads.make_decode_case(name, num_layers=3, num_q_heads=16, num_kv_heads=8,
                                      head_dim=128, page_size=1, batch=12, ctx_lo=1, ctx_hi=700,
                                      num_dummy=4, dummy_seq_len=1, min_rows=256, value_std=0.5,
                                      seed=zlib.crc32(name.encode()) % 10000)
    pool_t, k_new, v_new, q = workloads.make_decode_values(case, DEV)
    host_pool = [(gu.u16(pool_t[0, l]), gu.u16(pool_t[1, l])) for l in range(case.num_layers)]
    pool = mk.KVPool(pool_t, case.page_size)
    pt, sl, loc = case.page_table.to(DEV), case.seq_lens.to(DEV), case.out_loc.to(DEV)
    ws = mk.decode_workspace(case.batch, case.num_q_heads, pool)
    outs = [torch.empty_like(q[l]) for l in range(case.num_layers)]

    def step():
        for l in range(case.num_layers):
            mk.minisgl_store_decode_attn(pool, l, k_new[l], v_new[l], loc, q[l], pt, sl,
                                         case.sm_scale, out=outs[l], workspace=ws,
                                         split_tokens=split_tokens)

    step()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    orc = oracle.get()
    for l in range(case.num_layers):
        hk, hv = host_pool[l]
        orc.store_kv(hk, hv, k_new[l].cpu(), v_new[l].cpu(), case.out_loc)
        assert np.array_equal(gu.u16(pool_t[0, l]), hk)
        assert np.array_equal(gu.u16(pool_t[1, l]), hv)
        ref, _ = orc.decode(q[l].cpu(), hk, hv, case.page_table, case.seq_lens, case.sm_scale)
        real = case.num_real
        gu.check_attn(eager[l][:real], ref[:real], f"{name} layer {l}")

    g = _capture(step)
    for o in outs:
        o.fill_(0)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        for l in range(case.num_layers):
            assert torch.equal(outs[l], eager[l]), f"replayed layer {l} differs from eager"
    for l in range(case.num_layers):
        hk, hv = host_pool[l]
        assert np.array_equal(gu.u16(pool_t[0, l]), hk)
        assert np.array_equal(gu.u16(pool_t[1, l]), hv)


def test_graph_extend():
    case = workloads.make_extend_case("graph-extend", num_q_heads=8, num_kv_heads=2, head_dim=128,
                                      num_reqs=4, prefix_len=200, ext_lo=30, ext_hi=300,
                                      budget=4096, seed=4242)
    pool_t, per_batch = workloads.make_extend_values(case, DEV)
    pool = mk.KVPool(pool_t)
    b = case.batches[0]
    k, v, q = per_batch[0]
    args = [t.to(DEV) for t in (b.page_table, b.cached_lens, b.extend_lens, b.q_offsets, b.out_loc)]
    mk.minisgl_store_kv(pool, 0, k, v, args[4])
    out = torch.empty_like(q)

    def call():
        mk.minisgl_extend_attn(pool, 0, q, args[0], args[1], args[2], args[3], case.sm_scale,
                               out=out)

    call()
    torch.cuda.synchronize()
    eager = out.clone()
    g = _capture(call)
    out.fill_(0)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager), "replayed extend output differs from eager"
    assert mk.minisgl_debug_timeout_count() == 0


def test_graph_extend_with_caller_counter():
    """The extend call with the caller's own work counter, captured and replayed."""
    case = workloads.make_extend_case("graph-extend-ctr", num_q_heads=12, num_kv_heads=2, head_dim=64,
                                      num_reqs=3, prefix_len=150, ext_lo=30, ext_hi=300,
                                      budget=4096, seed=4243)
    pool_t, per_batch = workloads.make_extend_values(case, DEV)
    pool = mk.KVPool(pool_t)
    b = case.batches[0]
    k, v, q = per_batch[0]
    args = [t.to(DEV) for t in (b.page_table, b.cached_lens, b.extend_lens, b.q_offsets, b.out_loc)]
    mk.minisgl_store_kv(pool, 0, k, v, args[4])
    out = torch.empty_like(q)
    ctr = mk.extend_work_counter()

    def call():
        mk.minisgl_extend_attn(pool, 0, q, args[0], args[1], args[2], args[3], case.sm_scale,
                               out=out, work_counter=ctr)

    call()
    torch.cuda.synchronize()
    eager = out.clone()
    g = _capture(call)
    out.fill_(0)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager), "replayed extend output differs from eager"
    assert ctr.cpu().tolist() == [0, 0]
    assert mk.minisgl_debug_timeout_count() == 0


def test_graph_cascade_decode_and_extend():
    """Shared-prefix decode (its suffix part forked onto the library's second
    stream and joined back) and shared-prefix extend, captured in one graph
    and replayed: outputs equal the eager ones, and the eager ones match the
    oracle."""
    dc = workloads.decode_shared_prefix_qwen3(prefix_len=1024)
    dpool_t, k_new, v_new, dq = workloads.make_decode_values(dc, DEV)
    dpool = mk.KVPool(dpool_t)
    hk, hv = gu.u16(dpool_t[0, 0]), gu.u16(dpool_t[1, 0])
    dpt, dsl = dc.page_table.to(DEV), dc.seq_lens.to(DEV)
    mk.minisgl_store_kv(dpool, 0, k_new[0], v_new[0], dc.out_loc.to(DEV))
    dout = torch.empty_like(dq[0])
    ec = workloads.make_extend_case("graph-cascade-ext", num_q_heads=16, num_kv_heads=4, head_dim=128,
                                    num_reqs=4, prefix_len=300, ext_lo=30, ext_hi=300, budget=4096,
                                    seed=4244)
    epool_t, per_batch = workloads.make_extend_values(ec, DEV)
    epool = mk.KVPool(epool_t)
    eb = ec.batches[0]
    k, v, q = per_batch[0]
    eargs = [t.to(DEV) for t in (eb.page_table, eb.cached_lens, eb.extend_lens, eb.q_offsets, eb.out_loc)]
    mk.minisgl_store_kv(epool, 0, k, v, eargs[4])
    eout = torch.empty_like(q)

    def call():
        mk.minisgl_cascade_decode_attn(dpool, 0, dq[0], dpt, dsl, dc.shared_len, dc.sm_scale, out=dout)
        mk.minisgl_cascade_extend_attn(epool, 0, q, eargs[0], eargs[1], eargs[2], eargs[3], 300,
                                       ec.sm_scale, out=eout)

    call()
    torch.cuda.synchronize()
    d_eager, e_eager = dout.clone(), eout.clone()
    orc = oracle.get()
    orc.store_kv(hk, hv, k_new[0].cpu(), v_new[0].cpu(), dc.out_loc)
    ref, _ = gu.parallel_oracle_decode(hk, hv, dq[0], dc.page_table, dc.seq_lens, dc.sm_scale)
    gu.check_attn(d_eager, ref, "eager cascade decode")
    ehk, ehv = gu.u16(epool_t[0, 0]), gu.u16(epool_t[1, 0])
    eref = orc.extend(q.cpu(), ehk, ehv, eb.page_table, eb.cached_lens, eb.extend_lens, ec.sm_scale)
    gu.check_attn(e_eager, eref, "eager cascade extend")
    g = _capture(call)
    dout.fill_(0)
    eout.fill_(0)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(dout, d_eager), "replayed cascade decode differs from eager"
        assert torch.equal(eout, e_eager), "replayed cascade extend differs from eager"
    assert mk.minisgl_debug_timeout_count() == 0
