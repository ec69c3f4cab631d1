"""GPU parity of store_kv, split-KV decode and the LSE merge against the fp64 oracle.

Small cases are compared element by element; they span several 16-token
tiles, ragged tails, every supported group size, both head dims, 64-row pages,
CUDA-Graph padding requests, zero- and one-token contexts and forced split
counts.  All calls go through the C ABI (the ctypes binding).
"""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_row_gb300 as mk
import workloads
from tests import gpu_util as gu
from tests import oracle_pins

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_row_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def run_case(case, split_tokens=0, max_splits=16, layers=None, fused=False):
    """Store + decode every layer (fused: in one minisgl_store_decode_attn
    call); compare pool bytes and outputs with the oracle."""
    pool_t, k_new, v_new, q = workloads.make_decode_values(case, DEV)
    host_pool = [(gu.u16(pool_t[0, l]), gu.u16(pool_t[1, l])) for l in range(case.num_layers)]
    pool = mk.KVPool(pool_t, case.page_size)
    pt, sl, loc = case.page_table.to(DEV), case.seq_lens.to(DEV), case.out_loc.to(DEV)
    orc = oracle.get()
    outs = []
    for l in (layers or range(case.num_layers)):
        if fused:
            o = mk.minisgl_store_decode_attn(pool, l, k_new[l], v_new[l], loc, q[l], pt, sl,
                                             case.sm_scale, split_tokens=split_tokens,
                                             max_splits=max_splits)
        else:
            mk.minisgl_store_kv(pool, l, k_new[l], v_new[l], loc)
            o = mk.minisgl_decode_attn(pool, l, q[l], pt, sl, case.sm_scale,
                                       split_tokens=split_tokens, max_splits=max_splits)
        torch.cuda.synchronize()
        hk, hv = host_pool[l]
        orc.store_kv(hk, hv, k_new[l].cpu(), v_new[l].cpu(), case.out_loc)
        assert np.array_equal(gu.u16(pool_t[0, l]), hk), "K pool differs from oracle store_kv"
        assert np.array_equal(gu.u16(pool_t[1, l]), hv), "V pool differs from oracle store_kv"
        ref, _ = orc.decode(q[l].cpu(), hk, hv, case.page_table, case.seq_lens, case.sm_scale)
        gu.check_attn(o, ref, f"{case.name} layer {l}")
        outs.append(o)
    return outs, pool_t


SMALL = [
    # name, Hq, Hkv, d, page, B, ctx_lo, ctx_hi, dummies, layers
    ("g4-d64", 8, 2, 64, 1, 5, 1, 200, 0, 2),
    ("g2-d128", 16, 8, 128, 1, 6, 1, 300, 0, 1),
    ("g1-d128", 4, 4, 128, 1, 5, 1, 180, 0, 1),
    ("g16-d128", 32, 2, 128, 1, 3, 15, 150, 0, 1),
    ("g16-d64", 16, 1, 64, 1, 4, 1, 90, 0, 1),
    ("g8-page64", 64, 8, 128, 64, 3, 100, 700, 0, 1),
    ("g4-dummies", 32, 8, 128, 1, 8, 20, 260, 3, 1),
    ("g3-d128", 6, 2, 128, 1, 4, 1, 77, 0, 1),
]


@pytest.mark.parametrize("name,Hq,Hkv,d,page,B,lo,hi,dummies,L", SMALL, ids=[s[0] for s in SMALL])
def test_decode_small(name, Hq, Hkv, d, page, B, lo, hi, dummies, L):
    case = workloads.make_decode_case(name, num_layers=L, num_q_heads=Hq, num_kv_heads=Hkv,
                                      head_dim=d, page_size=page, batch=B, ctx_lo=lo, ctx_hi=hi,
                                      num_dummy=dummies, dummy_seq_len=9, min_rows=256,
                                      value_std=0.5, seed=zlib.crc32(name.encode()) % 10000)
    run_case(case)


@pytest.mark.parametrize("name,Hq,Hkv,d,page,B,lo,hi,dummies,L", SMALL, ids=[s[0] for s in SMALL])
def test_store_decode_fused_small(name, Hq, Hkv, d, page, B, lo, hi, dummies, L):
    """store_kv fused into decode: the same pool bytes and outputs as the
    two calls, on every small case (padding requests with 9-token contexts on
    the dummy row included)."""
    case = workloads.make_decode_case(name, num_layers=L, num_q_heads=Hq, num_kv_heads=Hkv,
                                      head_dim=d, page_size=page, batch=B, ctx_lo=lo, ctx_hi=hi,
                                      num_dummy=dummies, dummy_seq_len=9, min_rows=256,
                                      value_std=0.5, seed=zlib.crc32(name.encode()) % 10000)
    run_case(case, fused=True)


@pytest.mark.parametrize("split_tokens", [16, 48])
def test_store_decode_fused_split_counts(split_tokens):
    case = workloads.make_decode_case("fused-splits", num_layers=1, num_q_heads=16, num_kv_heads=4,
                                      head_dim=128, page_size=1, batch=5, ctx_lo=1, ctx_hi=400,
                                      value_std=0.5, seed=78)
    run_case(case, split_tokens=split_tokens, max_splits=64, fused=True)


def test_tiny_decode_config():
    """The tiny decode workload (batch 4, GQA 4, d 64, 4096-row pool), whole."""
    run_case(workloads.decode_tiny())


@pytest.mark.parametrize("split_tokens", [16, 32, 48, 112, 100000])
def test_split_counts(split_tokens):
    """Forced partial lengths (many splits per request down to one split):
    every setting matches the oracle, so the merge is right at each count."""
    case = workloads.make_decode_case("splits", num_layers=1, num_q_heads=16, num_kv_heads=4,
                                      head_dim=128, page_size=1, batch=5, ctx_lo=40, ctx_hi=400,
                                      value_std=0.5, seed=77)
    run_case(case, split_tokens=split_tokens, max_splits=64)


def test_partials_match_oracle_ranges():
    """The workspace partials (normalised o and natural-log lse per split)
    equal the oracle over each split's token range; the split boundaries follow
    the documented schedule: streams (request, KV head) of 16-token tiles laid
    end to end, cut into segments of split_tokens/16 tiles."""
    Hq, Hkv, d, S = 8, 2, 128, 64
    case = workloads.make_decode_case("partials", num_layers=1, num_q_heads=Hq, num_kv_heads=Hkv,
                                      head_dim=d, page_size=1, batch=4, ctx_lo=50, ctx_hi=300,
                                      value_std=0.5, seed=78)
    pool_t, k_new, v_new, q = workloads.make_decode_values(case, DEV)
    hk, hv = gu.u16(pool_t[0, 0]), gu.u16(pool_t[1, 0])
    pool = mk.KVPool(pool_t)
    B = case.batch
    ws = torch.zeros(mk.minisgl_decode_workspace_bytes(B, Hq, Hkv, d, S), dtype=torch.uint8, device=DEV)
    mk.minisgl_store_kv(pool, 0, k_new[0], v_new[0], case.out_loc.to(DEV))
    split = 48
    out = mk.minisgl_decode_attn(pool, 0, q[0], case.page_table.to(DEV), case.seq_lens.to(DEV),
                                 case.sm_scale, workspace=ws, split_tokens=split)
    torch.cuda.synchronize()
    orc = oracle.get()
    orc.store_kv(hk, hv, k_new[0].cpu(), v_new[0].cpu(), case.out_loc)
    al = lambda x: (x + 255) // 256 * 256
    raw = ws.cpu().numpy()
    counts = raw[:B * Hkv * 4].view(np.int32)
    off_lse = al(B * Hkv * 4)
    lse = raw[off_lse:off_lse + B * Hq * S * 4].view(np.float32).reshape(B, Hq, S)
    off_o = off_lse + al(B * Hq * S * 4)
    po = raw[off_o:off_o + B * Hq * S * d * 4].view(np.float32).reshape(B, Hq, S, d)
    # host replica of the schedule
    P = split // 16
    nt = [(int(n) + 15) // 16 for n in case.seq_lens]
    start, t = [], 0
    for r in range(B):
        start.append(t)
        t += nt[r] * Hkv
    G = Hq // Hkv
    checked = 0
    for r in range(B):
        for g in range(Hkv):
            s0 = start[r] + g * nt[r]
            s1 = s0 + nt[r]
            k0 = s0 // P
            nsplit = (s1 - 1) // P - k0 + 1
            assert counts[r * Hkv + g] == nsplit, (r, g, counts[r * Hkv + g], nsplit)
            if nsplit == 1:
                continue
            for s in range(nsplit):
                a = max(s0, (k0 + s) * P) - s0
                b = min(s1, (k0 + s + 1) * P) - s0
                jb = torch.tensor([a * 16], dtype=torch.int32)
                je = torch.tensor([min(b * 16, int(case.seq_lens[r]))], dtype=torch.int32)
                ro, rl = orc.decode(q[0, r:r + 1].cpu(), hk, hv, case.page_table[r:r + 1], je,
                                    case.sm_scale, j_begin=jb)
                for i in range(G):
                    h = g * G + i
                    assert abs(lse[r, h, s] - rl[0, h]) < 1e-3 * max(1, abs(rl[0, h])), (r, h, s)
                    assert np.abs(po[r, h, s] - ro[0, h]).max() < 1e-2
                checked += 1
    assert checked > 4
    ref, _ = orc.decode(q[0].cpu(), hk, hv, case.page_table, case.seq_lens, case.sm_scale)
    gu.check_attn(out, ref, "partials merged")


def test_split_invariance_and_determinism():
    case = workloads.make_decode_case("inv", num_layers=1, num_q_heads=16, num_kv_heads=8,
                                      head_dim=128, page_size=1, batch=7, ctx_lo=1, ctx_hi=500,
                                      value_std=0.5, seed=79)
    a, _ = run_case(case, split_tokens=0)
    b, _ = run_case(case, split_tokens=0)
    assert torch.equal(a[0], b[0]), "same inputs, same launch: output must be bit-identical"
    c, _ = run_case(case, split_tokens=32)
    err = (a[0].float() - c[0].float()).abs().max().item()
    assert err <= 2 * gu.MAX_ABS


def test_zero_and_one_token_contexts():
    """seq_len 0 gives zeros; seq_len 1 gives that token's V (rounded to bf16)."""
    Hq, Hkv, d, R = 8, 2, 128, 64
    g = torch.Generator().manual_seed(5)
    pool_t = (torch.randn((2, 1, R, Hkv, d), generator=g) * 0.5).to(torch.bfloat16).to(DEV)
    pool = mk.KVPool(pool_t)
    q = (torch.randn((3, Hq, d), generator=g)).to(torch.bfloat16).to(DEV)
    pt = torch.tensor([[5] + [R - 1] * 31, [R - 1] * 32, [9, 3] + [R - 1] * 30], dtype=torch.int32, device=DEV)
    sl = torch.tensor([1, 0, 2], dtype=torch.int32, device=DEV)
    out = mk.minisgl_decode_attn(pool, 0, q, pt, sl, 0.1)
    torch.cuda.synchronize()
    G = Hq // Hkv
    for h in range(Hq):
        assert torch.equal(out[0, h], pool_t[1, 0, 5, h // G]), "1-token context must return V"
    assert torch.count_nonzero(out[1]) == 0, "empty context must give zeros"


def test_permutation_invariance_bitwise():
    """Relabelling physical rows (and the page table with them) leaves the
    GPU output bit-identical: the reduction order depends on logical order only."""
    case = workloads.make_decode_case("perm", num_layers=1, num_q_heads=16, num_kv_heads=8,
                                      head_dim=128, page_size=1, batch=5, ctx_lo=1, ctx_hi=300,
                                      value_std=0.5, seed=80)
    pool_t, _, _, q = workloads.make_decode_values(case, DEV)
    perm = torch.randperm(case.num_rows, generator=torch.Generator().manual_seed(3)).to(DEV)
    pool2 = torch.empty_like(pool_t)
    pool2[:, :, perm] = pool_t
    pt = case.page_table.to(DEV)
    pt2 = perm[pt.long()].to(torch.int32)
    sl = case.seq_lens.to(DEV)
    a = mk.minisgl_decode_attn(mk.KVPool(pool_t), 0, q[0], pt, sl, case.sm_scale)
    b = mk.minisgl_decode_attn(mk.KVPool(pool2), 0, q[0], pt2, sl, case.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_page_table_example_golden():
    """The pages' page-table example (requests A, B, Seq1, Seq2), embedded in
    head_dim 64 with zero padding, against the hand-derived closed forms."""
    import json, os
    fx = json.load(open(os.path.join(oracle_pins.GOLDEN, "page_table_example.json")))
    d = 64
    K = torch.zeros((7, 1, d), dtype=torch.float64)
    V = torch.zeros((7, 1, d), dtype=torch.float64)
    K[:, 0, :2] = torch.tensor(fx["K"], dtype=torch.float64)
    V[:, 0, :2] = torch.tensor(fx["V"], dtype=torch.float64)
    R = 8
    pool_t = torch.zeros((2, 1, R, 1, d), dtype=torch.bfloat16)
    pool_t[0, 0, :7] = K.to(torch.bfloat16)
    pool_t[1, 0, :7] = V.to(torch.bfloat16)
    pool_t[:, 0, 7] = float("nan")  # padding columns point here
    pt = torch.full((4, 32), 7, dtype=torch.int32)
    for r, rows in enumerate(fx["page_table"]):
        pt[r, :len(rows)] = torch.tensor(rows, dtype=torch.int32)
    sl = torch.tensor([len(x) for x in fx["page_table"]], dtype=torch.int32)
    q = torch.zeros((4, 1, d), dtype=torch.float64)
    q[:, 0, :2] = torch.tensor(fx["q"], dtype=torch.float64)
    scale = math.log(3) / 2
    out = mk.minisgl_decode_attn(mk.KVPool(pool_t.to(DEV)), 0, q.to(torch.bfloat16).to(DEV),
                                 pt.to(DEV), sl.to(DEV), scale)
    torch.cuda.synchronize()
    ev = lambda e: float(eval(e, {"__builtins__": {}}, {"log": math.log, "sqrt": math.sqrt}))
    exp = np.zeros((4, 1, d))
    exp[:, 0, :2] = [[ev(e) for e in row] for row in fx["expected_out"]]
    gu.check_attn(out, exp, "page-table example")


def test_store_kv_strided_and_pagefirst():
    """store_kv on a PageFirst pool (pages outermost, permuted view) with k/v
    taken as strided slices of a fused qkv buffer; other layers untouched."""
    L, R, Hkv, d, N, Hq = 3, 300, 2, 128, 9, 8
    g = torch.Generator().manual_seed(8)
    base = (torch.randn((2, R, L, Hkv, d), generator=g) * 0.5).to(torch.bfloat16).to(DEV)
    pool_t = base.permute(0, 2, 1, 3, 4)  # logical (2, L, R, Hkv, d)
    pool = mk.KVPool(pool_t)
    qkv = (torch.randn((N, Hq + 2 * Hkv, d), generator=g) * 0.5).to(torch.bfloat16).to(DEV)
    k, v = qkv[:, Hq:Hq + Hkv], qkv[:, Hq + Hkv:]
    loc = torch.randperm(R - 1, generator=g)[:N].to(torch.int32)
    before = [gu.u16(pool_t[0, l].contiguous()) for l in range(L)]
    mk.minisgl_store_kv(pool, 1, k, v, loc.to(DEV))
    torch.cuda.synchronize()
    exp_k = pool_t[0, 1].cpu().clone()
    exp_k[:] = torch.from_numpy(before[1].view(np.int16)).view(torch.bfloat16)
    exp_k[loc.long()] = k.cpu()
    assert torch.equal(pool_t[0, 1].cpu(), exp_k)
    assert torch.equal(pool_t[1, 1].cpu()[loc.long()], v.cpu())
    for l in (0, 2):
        assert np.array_equal(gu.u16(pool_t[0, l].contiguous()), before[l]), "other layers must not change"


@pytest.mark.parametrize("split_tokens", [0, 16])
def test_large_batch_short_contexts(split_tokens):
    """1040 requests x 8 KV heads = 8320 (request, KV head) streams of at most
    4 tiles: many streams per warp at the automatic split, and with forced
    16-token splits nearly every stream is split and merged."""
    case = workloads.make_decode_case("many-streams", num_layers=1, num_q_heads=8, num_kv_heads=8,
                                      head_dim=64, page_size=1, batch=1040, ctx_lo=1, ctx_hi=60,
                                      value_std=0.5, seed=81)
    run_case(case, split_tokens=split_tokens, max_splits=16)


@pytest.mark.parametrize("fused", [False, True])
def test_decode_max_batch(fused):
    """The largest batch the call accepts (4,096 requests), short contexts:
    the per-request schedule prefix fills 16 KB of shared memory."""
    case = workloads.make_decode_case("max-batch", num_layers=1, num_q_heads=8, num_kv_heads=2,
                                      head_dim=128, page_size=1, batch=4096, ctx_lo=1, ctx_hi=24,
                                      value_std=0.5, seed=82)
    run_case(case, fused=fused)
