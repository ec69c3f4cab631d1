"""GPU parity of the tcgen05 causal extend kernel against the fp64 oracle.

Cases span several 128-token KV tiles and several query blocks with ragged
tails, every supported group size, empty and one-token prefixes and extends,
radix-shared prefix rows and chunked-prefill batches whose later chunks read
rows stored by earlier ones.
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


def run_extend_case(case, check=True):
    """store_kv + extend for every batch in order, against the oracle doing the same."""
    pool_t, per_batch = workloads.make_extend_values(case, DEV)
    hk, hv = gu.u16(pool_t[0, 0]), gu.u16(pool_t[1, 0])
    pool = mk.KVPool(pool_t)
    orc = oracle.get()
    outs = []
    for b, (k, v, q) in zip(case.batches, per_batch):
        mk.minisgl_store_kv(pool, 0, k, v, b.out_loc.to(DEV))
        o = mk.minisgl_extend_attn(pool, 0, q, b.page_table.to(DEV), b.cached_lens.to(DEV),
                                   b.extend_lens.to(DEV), b.q_offsets.to(DEV), case.sm_scale)
        torch.cuda.synchronize()
        orc.store_kv(hk, hv, k.cpu(), v.cpu(), b.out_loc)
        if check:
            assert np.array_equal(gu.u16(pool_t[0, 0]), hk), "K pool differs from oracle store_kv"
            ref = orc.extend(q.cpu(), hk, hv, b.page_table, b.cached_lens, b.extend_lens,
                             case.sm_scale)
            gu.check_attn(o, ref, f"{case.name} batch {len(outs)}")
        outs.append(o)
    assert mk.minisgl_debug_timeout_count() == 0, "a tensor-core kernel wait ran out"
    return outs


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 7, 8, 12, 16])
def test_extend_head_dims_and_group_sizes(G, d):
    """Every group size 1..8 (and 12, 16) at head_dim 64 and 128.  Groups that
    do not divide 128 leave dead MMA rows past floor(128/G)*G in each tile."""
    Hkv = 2
    case = workloads.make_extend_case(f"g{G}-d{d}", num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=d,
                                      num_reqs=3, prefix_len=70, ext_lo=1, ext_hi=260, budget=4096,
                                      seed=300 + G + d)
    run_extend_case(case)


def _manual_case(cached, ext, Hq=8, Hkv=2, seed=0, d=128):
    """Requests with given cached / extend lengths, private rows, one batch."""
    g = torch.Generator().manual_seed(seed)
    lens = [c + e for c, e in zip(cached, ext)]
    R = sum(lens) + 40
    perm = torch.randperm(R - 2, generator=g).to(torch.int32)
    W = workloads.align_up(max(lens + [1]))
    pt = torch.full((len(lens), W), R - 1, dtype=torch.int32)
    outs = []
    off = 0
    for r, n in enumerate(lens):
        pt[r, :n] = perm[off:off + n]
        outs.append(perm[off + cached[r]:off + n])
        off += n
    qo = torch.zeros(len(lens) + 1, dtype=torch.int32)
    qo[1:] = torch.cumsum(torch.tensor(ext, dtype=torch.int32), 0)
    case = workloads.ExtendCase(name="manual", num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                                num_rows=R, prefix_rows=perm[:0], extend_lens=list(ext),
                                sm_scale=1 / d ** 0.5, value_std=0.5, seed=seed)
    case.batches.append(workloads.ExtendBatch(
        req_ids=list(range(len(lens))), cached_lens=torch.tensor(cached, dtype=torch.int32),
        extend_lens=torch.tensor(ext, dtype=torch.int32), q_offsets=qo, page_table=pt,
        out_loc=torch.cat(outs).to(torch.int32)))
    return case


@pytest.mark.parametrize("Hq,Hkv,d", [(8, 2, 128), (6, 2, 64), (14, 2, 128)])
def test_extend_edge_lengths(Hq, Hkv, d):
    """No prefix, one-token extends, extends ending exactly on tile edges and
    on query-tile edges (42 tokens per tile at group 3, 18 at group 7),
    prefixes ending on tile edges, and an empty extend in the middle."""
    cached = [0, 0, 128, 5, 127, 300, 0, 256, 0, 10]
    ext = [1, 128, 1, 0, 129, 33, 257, 64, 42, 85]
    run_extend_case(_manual_case(cached, ext, Hq=Hq, Hkv=Hkv, seed=41, d=d))


def test_extend_caller_counters_on_two_streams():
    """Two extend calls at a time on two unordered streams, each with its own
    work counter, three rounds: both match the oracle and both counters are
    back at zero afterwards."""
    cases = [_manual_case([300, 0, 900], [700, 513, 260], Hq=32, Hkv=8, seed=61),
             _manual_case([0, 1500], [1000, 300], Hq=32, Hkv=8, seed=62)]
    orc = oracle.get()
    runs = []
    for case in cases:
        pool_t, per_batch = workloads.make_extend_values(case, DEV)
        hk, hv = gu.u16(pool_t[0, 0]), gu.u16(pool_t[1, 0])
        pool = mk.KVPool(pool_t)
        b = case.batches[0]
        k, v, q = per_batch[0]
        mk.minisgl_store_kv(pool, 0, k, v, b.out_loc.to(DEV))
        orc.store_kv(hk, hv, k.cpu(), v.cpu(), b.out_loc)
        args = (b.page_table.to(DEV), b.cached_lens.to(DEV), b.extend_lens.to(DEV), b.q_offsets.to(DEV))
        runs.append((case, pool, q, args, torch.empty_like(q), mk.extend_work_counter(), (hk, hv)))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for _ in range(3):
        for (case, pool, q, args, out, ctr, _), st in zip(runs, streams):
            with torch.cuda.stream(st):
                mk.minisgl_extend_attn(pool, 0, q, *args, case.sm_scale, out=out, work_counter=ctr)
    torch.cuda.synchronize()
    for case, pool, q, args, out, ctr, (hk, hv) in runs:
        b = case.batches[0]
        ref = orc.extend(q.cpu(), hk, hv, b.page_table, b.cached_lens, b.extend_lens, case.sm_scale)
        gu.check_attn(out, ref, "extend with a caller counter")
        assert ctr.cpu().tolist() == [0, 0], "work counter not left at zero"
    assert mk.minisgl_debug_timeout_count() == 0


def test_extend_mixed_chunk_and_decode_batch():
    """One extend launch carrying chunked-prefill requests and decode requests
    (one new token over a long context) side by side, as a mixed batch does."""
    g = torch.Generator().manual_seed(77)
    n_dec = 24
    cached = [0, 300, 1100] + torch.randint(100, 3000, (n_dec,), generator=g).tolist()
    ext = [400, 257, 129] + [1] * n_dec
    run_extend_case(_manual_case(cached, ext, Hq=32, Hkv=8, seed=78))


def test_extend_growing_scores_take_the_exact_path():
    """Scores that jump by far more than the rescale threshold from one
    128-token K/V tile to the next: the running-max fast path must hand such
    tiles to the exact path (and rescale O); results still match the oracle."""
    case = _manual_case([600, 0], [80, 300], Hq=8, Hkv=2, seed=12)
    pool_t, per_batch = workloads.make_extend_values(case, DEV)
    b = case.batches[0]
    k, v, q = per_batch[0]
    g = torch.Generator(device=DEV).manual_seed(3)
    levels = torch.tensor([0.05, 0.6, 1.6, 3.4, 6.0], device=DEV)

    def keys(pos):  # key value grows with the position's 128-token tile
        f = levels[(pos // 128).clamp(max=4)]
        noise = torch.randn((pos.numel(), 2, 128), generator=g, device=DEV) * 0.02
        return (f[:, None, None] + noise).to(torch.bfloat16)

    for r, (C, E) in enumerate(zip(b.cached_lens.tolist(), b.extend_lens.tolist())):
        o = int(b.q_offsets[r])
        if C:
            rows = b.page_table[r, :C].long().to(DEV)
            pool_t[0, 0, rows] = keys(torch.arange(C, device=DEV))
        k[o:o + E] = keys(torch.arange(C, C + E, device=DEV))
    q.copy_((0.5 + 0.05 * torch.randn(q.shape, generator=g, device=DEV)).to(torch.bfloat16))
    hk, hv = gu.u16(pool_t[0, 0]), gu.u16(pool_t[1, 0])
    pool = mk.KVPool(pool_t)
    mk.minisgl_store_kv(pool, 0, k, v, b.out_loc.to(DEV))
    o = mk.minisgl_extend_attn(pool, 0, q, b.page_table.to(DEV), b.cached_lens.to(DEV),
                               b.extend_lens.to(DEV), b.q_offsets.to(DEV), case.sm_scale)
    torch.cuda.synchronize()
    orc = oracle.get()
    orc.store_kv(hk, hv, k.cpu(), v.cpu(), b.out_loc)
    ref = orc.extend(q.cpu(), hk, hv, b.page_table, b.cached_lens, b.extend_lens, case.sm_scale)
    gu.check_attn(o, ref, "growing scores")
    assert mk.minisgl_debug_timeout_count() == 0


def test_extend_prefix_shared_equals_private():
    """Requests pointing at one set of radix-cache prefix rows give bit-identical
    output to requests holding private copies of the same values."""
    kw = dict(num_q_heads=16, num_kv_heads=4, head_dim=128, num_reqs=4, prefix_len=300,
              ext_lo=50, ext_hi=200, budget=8192, seed=91)
    shared = workloads.make_extend_case("shared", **kw)
    private = workloads.make_extend_case("private", shared_prefix=False, **kw)
    assert shared.extend_lens == private.extend_lens
    pool_s, pb = workloads.make_extend_values(shared, DEV)
    # private pool: same values at the private prefix rows and the new rows
    pool_p = torch.zeros((2, 1, private.num_rows, 4, 128), dtype=torch.bfloat16, device=DEV)
    for rs, rp in zip([shared.prefix_rows] * 4, private.prefix_rows_per_req):
        pool_p[:, 0, rp.long().to(DEV)] = pool_s[:, 0, rs.long().to(DEV)]
    outs = []
    for case, pool_t in ((shared, pool_s), (private, pool_p)):
        pool = mk.KVPool(pool_t)
        o = []
        for b, (k, v, q) in zip(case.batches, pb):
            mk.minisgl_store_kv(pool, 0, k, v, b.out_loc.to(DEV))
            o.append(mk.minisgl_extend_attn(pool, 0, q, b.page_table.to(DEV), b.cached_lens.to(DEV),
                                            b.extend_lens.to(DEV), b.q_offsets.to(DEV),
                                            case.sm_scale))
        outs.append(o)
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_extend_chunked_batches():
    """Chunked prefill: a request cut by the token budget continues in the next
    batch and reads the rows its first chunk stored."""
    case = workloads.make_extend_case("chunked", num_q_heads=8, num_kv_heads=2, head_dim=128,
                                      num_reqs=5, prefix_len=100, ext_lo=60, ext_hi=300,
                                      budget=256, seed=17)
    assert len(case.batches) >= 3
    assert any(int(b.cached_lens[0]) > 100 for b in case.batches[1:]), "expect a continued chunk"
    run_extend_case(case)


def test_extend_matches_decode_on_last_token():
    """The last new token of an extend equals a decode of the same query over
    the whole context (both kernels, same pool)."""
    case = _manual_case([200, 37], [50, 91], Hq=16, Hkv=8, seed=5)
    pool_t, per_batch = workloads.make_extend_values(case, DEV)
    pool = mk.KVPool(pool_t)
    b = case.batches[0]
    k, v, q = per_batch[0]
    mk.minisgl_store_kv(pool, 0, k, v, b.out_loc.to(DEV))
    o = mk.minisgl_extend_attn(pool, 0, q, b.page_table.to(DEV), b.cached_lens.to(DEV),
                               b.extend_lens.to(DEV), b.q_offsets.to(DEV), case.sm_scale)
    last = (b.q_offsets[1:] - 1).long()
    qd = q[last.to(DEV)].contiguous()
    seq = (b.cached_lens + b.extend_lens).to(DEV)
    od = mk.minisgl_decode_attn(pool, 0, qd, b.page_table.to(DEV), seq, case.sm_scale)
    torch.cuda.synchronize()
    err = (o[last.to(DEV)].float() - od.float()).abs().max().item()
    assert err <= 2 * gu.MAX_ABS


def _pagefirst(layer_pool, L, layer, seed):
    """A PageFirst pool (2, R, L, H_kv, d) in memory, seen as the logical
    (2, L, R, H_kv, d) view, whose `layer` holds the generator's values of a
    one-layer pool; the other layers hold other values."""
    _, _, R, Hkv, d = layer_pool.shape
    g = torch.Generator(device=DEV).manual_seed(seed)
    base = torch.empty((2, R, L, Hkv, d), dtype=torch.bfloat16, device=DEV).normal_(0, 0.5, generator=g)
    view = base.permute(0, 2, 1, 3, 4)
    view[:, layer] = layer_pool[:, 0]
    return view


def test_extend_and_decode_on_pagefirst_pool():
    """Extend and decode read a PageFirst pool (row stride L*H_kv*d, layer
    stride H_kv*d) through the same descriptor: results match the oracle on
    the layer's rows, and store_kv lands in that layer only."""
    L, layer = 3, 1
    case = workloads.make_extend_case("pagefirst-ext", num_q_heads=16, num_kv_heads=4, head_dim=128,
                                      num_reqs=3, prefix_len=150, ext_lo=40, ext_hi=230,
                                      budget=512, seed=31)
    pool1, per_batch = workloads.make_extend_values(case, DEV)
    pool_t = _pagefirst(pool1, L, layer, 32)
    assert pool_t.stride(2) == L * 4 * 128 and pool_t.stride(1) == 4 * 128
    hk, hv = gu.u16(pool1[0, 0]), gu.u16(pool1[1, 0])
    others = [gu.u16(pool_t[0, l]) for l in range(L) if l != layer]
    pool = mk.KVPool(pool_t)
    orc = oracle.get()
    for b, (k, v, q) in zip(case.batches, per_batch):
        mk.minisgl_store_kv(pool, layer, k, v, b.out_loc.to(DEV))
        o = mk.minisgl_extend_attn(pool, layer, q, b.page_table.to(DEV), b.cached_lens.to(DEV),
                                   b.extend_lens.to(DEV), b.q_offsets.to(DEV), case.sm_scale)
        torch.cuda.synchronize()
        orc.store_kv(hk, hv, k.cpu(), v.cpu(), b.out_loc)
        assert np.array_equal(gu.u16(pool_t[0, layer]), hk)
        ref = orc.extend(q.cpu(), hk, hv, b.page_table, b.cached_lens, b.extend_lens, case.sm_scale)
        gu.check_attn(o, ref, "pagefirst extend")
    now = [gu.u16(pool_t[0, l]) for l in range(L) if l != layer]
    assert all(a.tobytes() == b.tobytes() for a, b in zip(now, others)), "other layers changed"

    dcase = workloads.make_decode_case("pagefirst-dec", num_layers=1, num_q_heads=16, num_kv_heads=4,
                                       head_dim=128, page_size=1, batch=6, ctx_lo=20, ctx_hi=600,
                                       value_std=0.5, seed=33)
    dpool1, k_new, v_new, q = workloads.make_decode_values(dcase, DEV)
    dpool_t = _pagefirst(dpool1, L, layer, 34)
    dk, dv = gu.u16(dpool1[0, 0]), gu.u16(dpool1[1, 0])
    dpool = mk.KVPool(dpool_t)
    mk.minisgl_store_kv(dpool, layer, k_new[0], v_new[0], dcase.out_loc.to(DEV))
    out = mk.minisgl_decode_attn(dpool, layer, q[0], dcase.page_table.to(DEV), dcase.seq_lens.to(DEV),
                                 dcase.sm_scale)
    torch.cuda.synchronize()
    orc.store_kv(dk, dv, k_new[0].cpu(), v_new[0].cpu(), dcase.out_loc)
    ref, _ = orc.decode(q[0].cpu(), dk, dv, dcase.page_table, dcase.seq_lens, dcase.sm_scale)
    gu.check_attn(out, ref, "pagefirst decode")
    assert mk.minisgl_debug_timeout_count() == 0


@pytest.mark.parametrize("Hq,Hkv,d,P", [(8, 2, 128, 300), (32, 8, 128, 1000), (6, 2, 64, 129),
                                         (14, 2, 64, 64), (16, 16, 128, 1)])
def test_cascade_extend_matches_oracle(Hq, Hkv, d, P):
    """Shared-prefix extend over chunked batches: a request cut by the budget
    continues with cached_len > P; prefixes shorter than, equal to and longer
    than one tile, one shared position, head_dim 64, odd groups."""
    case = workloads.make_extend_case(f"cascade-ext-g{Hq // Hkv}-d{d}-p{P}", num_q_heads=Hq,
                                      num_kv_heads=Hkv, head_dim=d, num_reqs=5, prefix_len=P,
                                      ext_lo=1, ext_hi=400, budget=300, seed=500 + P + d)
    assert len(case.batches) >= 2
    pool_t, per_batch = workloads.make_extend_values(case, DEV)
    hk, hv = gu.u16(pool_t[0, 0]), gu.u16(pool_t[1, 0])
    pool = mk.KVPool(pool_t)
    orc = oracle.get()
    for bi, (b, (k, v, q)) in enumerate(zip(case.batches, per_batch)):
        mk.minisgl_store_kv(pool, 0, k, v, b.out_loc.to(DEV))
        o = mk.minisgl_cascade_extend_attn(pool, 0, q, b.page_table.to(DEV), b.cached_lens.to(DEV),
                                           b.extend_lens.to(DEV), b.q_offsets.to(DEV), P, case.sm_scale)
        torch.cuda.synchronize()
        orc.store_kv(hk, hv, k.cpu(), v.cpu(), b.out_loc)
        ref = orc.extend(q.cpu(), hk, hv, b.page_table, b.cached_lens, b.extend_lens, case.sm_scale)
        gu.check_attn(o, ref, f"{case.name} batch {bi}")
    assert mk.minisgl_debug_timeout_count() == 0


def test_extend_maximum_batch():
    """4096 requests (the largest batch the call takes; the per-request item
    prefix fills 16 KB of shared memory) of 0-40 cached and 1-3 new tokens,
    group size 4, against the oracle on every token."""
    g = torch.Generator().manual_seed(4096)
    B = 4096
    cached = torch.randint(0, 41, (B,), generator=g).tolist()
    ext = torch.randint(1, 4, (B,), generator=g).tolist()
    case = _manual_case(cached, ext, Hq=16, Hkv=4, seed=4097)
    b = case.batches[0]
    pool_t, per_batch = workloads.make_extend_values(case, DEV)
    hk, hv = gu.u16(pool_t[0, 0]), gu.u16(pool_t[1, 0])
    k, v, q = per_batch[0]
    pool = mk.KVPool(pool_t)
    mk.minisgl_store_kv(pool, 0, k, v, b.out_loc.to(DEV))
    o = mk.minisgl_extend_attn(pool, 0, q, b.page_table.to(DEV), b.cached_lens.to(DEV),
                               b.extend_lens.to(DEV), b.q_offsets.to(DEV), case.sm_scale)
    torch.cuda.synchronize()
    oracle.get().store_kv(hk, hv, k.cpu(), v.cpu(), b.out_loc)
    ref = gu.parallel_oracle_extend(hk, hv, q, b.page_table, b.cached_lens, b.extend_lens, b.q_offsets,
                                    case.sm_scale)
    gu.check_attn(o, ref, "extend, 4096 requests")
    assert mk.minisgl_debug_timeout_count() == 0


def test_page_table_row_stride_wider_than_width():
    """Page tables that are a column slice of a wider buffer (row stride
    larger than the width the call reads), for extend, decode and cascade
    decode: the same results as with the compact table, bit for bit."""
    case = _manual_case([100, 0, 333], [60, 200, 45], Hq=8, Hkv=2, seed=88)
    b = case.batches[0]
    pool_t, per_batch = workloads.make_extend_values(case, DEV)
    k, v, q = per_batch[0]
    pool = mk.KVPool(pool_t)
    mk.minisgl_store_kv(pool, 0, k, v, b.out_loc.to(DEV))
    W = b.page_table.shape[1]
    wide = torch.full((b.page_table.shape[0], W + 96), -7, dtype=torch.int32)
    wide[:, 16:16 + W] = b.page_table
    pt_view = wide.to(DEV)[:, 16:16 + W]  # stride W + 96, width W
    assert pt_view.stride(0) == W + 96 and pt_view.stride(1) == 1
    args = [t.to(DEV) for t in (b.cached_lens, b.extend_lens, b.q_offsets)]
    o1 = mk.minisgl_extend_attn(pool, 0, q, b.page_table.to(DEV), *args, case.sm_scale)
    o2 = mk.minisgl_extend_attn(pool, 0, q, pt_view, *args, case.sm_scale)
    seq = (b.cached_lens + b.extend_lens).to(DEV)
    qd = q[(b.q_offsets[1:] - 1).long().to(DEV)].contiguous()
    d1 = mk.minisgl_decode_attn(pool, 0, qd, b.page_table.to(DEV), seq, case.sm_scale)
    d2 = mk.minisgl_decode_attn(pool, 0, qd, pt_view, seq, case.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(d1, d2)
    sc = workloads.make_shared_prefix_decode_case("stride-cascade", num_q_heads=8, num_kv_heads=2, head_dim=128,
                                                  batch=7, prefix_len=300, suffix_lo=1, suffix_hi=90, seed=89)
    spool_t, sk, sv, sq = workloads.make_decode_values(sc, DEV)
    spool = mk.KVPool(spool_t)
    mk.minisgl_store_kv(spool, 0, sk[0], sv[0], sc.out_loc.to(DEV))
    SW = sc.page_table.shape[1]
    swide = torch.full((sc.batch, SW + 64), -7, dtype=torch.int32)
    swide[:, :SW] = sc.page_table
    sview = swide.to(DEV)[:, :SW]
    c1 = mk.minisgl_cascade_decode_attn(spool, 0, sq[0], sc.page_table.to(DEV), sc.seq_lens.to(DEV), 300,
                                        sc.sm_scale)
    c2 = mk.minisgl_cascade_decode_attn(spool, 0, sq[0], sview, sc.seq_lens.to(DEV), 300, sc.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)
    assert mk.minisgl_debug_timeout_count() == 0
