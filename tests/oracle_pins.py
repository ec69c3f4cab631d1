"""Pins for the fp64 oracle: checks against facts that do not come from the oracle.

Each pin takes an oracle instance (oracle.Oracle) and raises AssertionError when
the oracle disagrees with:
  * a closed form (one-token context returns V; equal scores return the mean of
    V and lse = log n; store_kv equals a library index_put);
  * a library routine on the same data (torch scaled_dot_product_attention in
    float64, with its own causal mask where the alignment coincides);
  * an invariant the pages fix (physical row order does not matter; a page
    table with 64-row pages reads the same values as one with single rows;
    requests sharing radix-cache prefix rows equal requests with private
    copies; CUDA-Graph padding requests touch only the dummy row);
  * values printed in the golden fixtures under tests/golden/;
  * for RoPE: position 0 is the identity, the rotation equals complex
    multiplication by exp(1j*theta) (numpy), and scores depend only on the
    relative position.
They are kept apart from the test functions so tests/test_oracle_mutations.py
can run the same pins against deliberately broken copies of the oracle and
check that every planted mistake is caught.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def bf16(x) -> torch.Tensor:
    return torch.as_tensor(x, dtype=torch.float64).to(torch.bfloat16)


def rnd(shape, g, std=1.0) -> torch.Tensor:
    return (torch.randn(shape, generator=g, dtype=torch.float64) * std).to(torch.bfloat16)


def f64(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.float64)


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def _random_decode(g, B=3, Hq=8, Hk=2, d=16, n_lo=1, n_hi=21, R=160, W=32):
    """Small random decode problem; padding page-table columns point at a NaN row."""
    pool_k = rnd((R, Hk, d), g)
    pool_v = rnd((R, Hk, d), g)
    poison = R - 1
    pool_k[poison] = float("nan")
    pool_v[poison] = float("nan")
    perm = torch.randperm(R - 1, generator=g)
    seq = torch.randint(n_lo, n_hi + 1, (B,), generator=g).to(torch.int32)
    pt = torch.full((B, W), poison, dtype=torch.int32)
    off = 0
    for r in range(B):
        n = int(seq[r])
        pt[r, :n] = perm[off:off + n].to(torch.int32)
        off += n
    q = rnd((B, Hq, d), g)
    return q, pool_k, pool_v, pt, seq


def _sdpa(qv, K, V, scale, mask=None, causal=False):
    """qv [Hq, Tq, d], K/V [Hk, n, d] float64 -> [Hq, Tq, d] through torch's SDPA."""
    G = qv.shape[0] // K.shape[0]
    K = K.repeat_interleave(G, dim=0)
    V = V.repeat_interleave(G, dim=0)
    return F.scaled_dot_product_attention(qv, K, V, attn_mask=mask, is_causal=causal, scale=scale)


# --------------------------------------------------------------------------- #
# store_kv
# --------------------------------------------------------------------------- #
def pin_store_kv_index_put(orc):
    g = torch.Generator().manual_seed(11)
    R, Hk, d, N = 96, 2, 8, 13
    pool_k, pool_v = rnd((R, Hk, d), g), rnd((R, Hk, d), g)
    k, v = rnd((N, Hk, d), g), rnd((N, Hk, d), g)
    loc = torch.randperm(R, generator=g)[:N].to(torch.int32)
    ok, ov = u16(pool_k), u16(pool_v)
    orc.store_kv(ok, ov, k, v, loc)
    ek, ev = pool_k.clone(), pool_v.clone()
    ek[loc.long()] = k  # library index_put
    ev[loc.long()] = v
    assert np.array_equal(ok, u16(ek)), "store_kv K differs from index_put"
    assert np.array_equal(ov, u16(ev)), "store_kv V differs from index_put"


# --------------------------------------------------------------------------- #
# decode
# --------------------------------------------------------------------------- #
def pin_single_token_returns_v(orc):
    g = torch.Generator().manual_seed(12)
    q, pk, pv, pt, _ = _random_decode(g)
    seq = torch.ones(q.shape[0], dtype=torch.int32)
    out, lse = orc.decode(q, pk, pv, pt, seq, 0.37)
    G = q.shape[1] // pk.shape[1]
    for r in range(q.shape[0]):
        row = int(pt[r, 0])
        for h in range(q.shape[1]):
            assert np.array_equal(out[r, h], f64(pv[row, h // G]).numpy()), "1-token ctx != V"
            s = 0.37 * float(np.dot(f64(q[r, h]).numpy(), f64(pk[row, h // G]).numpy()))
            assert abs(lse[r, h] - s) <= 1e-12 * max(1.0, abs(s)), "1-token lse != score"


def pin_equal_scores_mean(orc):
    g = torch.Generator().manual_seed(13)
    q, pk, pv, pt, seq = _random_decode(g, n_lo=3)
    G = q.shape[1] // pk.shape[1]
    # (a) zero query: every score is 0
    out, lse = orc.decode(torch.zeros_like(q), pk, pv, pt, seq, 0.5)
    for r in range(q.shape[0]):
        n = int(seq[r])
        rows = pt[r, :n].long()
        for h in range(q.shape[1]):
            mean = f64(pv[rows, h // G]).numpy().mean(axis=0)
            assert np.abs(out[r, h] - mean).max() <= 1e-13, "q=0 is not mean(V)"
            assert abs(lse[r, h] - math.log(n)) <= 1e-13, "q=0 lse != log n"
    # (b) identical keys, random query
    pk2 = pk.clone()
    for r in range(q.shape[0]):
        n = int(seq[r])
        pk2[pt[r, :n].long()] = pk[pt[r, 0].long()]
    out2, _ = orc.decode(q, pk2, pv, pt, seq, 0.5)
    for r in range(q.shape[0]):
        n = int(seq[r])
        rows = pt[r, :n].long()
        for h in range(q.shape[1]):
            mean = f64(pv[rows, h // G]).numpy().mean(axis=0)
            assert np.abs(out2[r, h] - mean).max() <= 1e-13, "equal keys is not mean(V)"


def pin_decode_matches_sdpa(orc):
    for seed, (Hq, Hk, d) in [(14, (8, 2, 16)), (15, (6, 6, 8)), (16, (8, 1, 32))]:
        g = torch.Generator().manual_seed(seed)
        q, pk, pv, pt, seq = _random_decode(g, Hq=Hq, Hk=Hk, d=d)
        scale = 1.0 / math.sqrt(d)
        out, lse = orc.decode(q, pk, pv, pt, seq, scale)
        for r in range(q.shape[0]):
            n = int(seq[r])
            rows = pt[r, :n].long()
            K = f64(pk[rows]).permute(1, 0, 2)  # [Hk, n, d]
            V = f64(pv[rows]).permute(1, 0, 2)
            qv = f64(q[r]).unsqueeze(1)           # [Hq, 1, d]
            ref = _sdpa(qv, K, V, scale)[:, 0]
            assert torch.allclose(torch.from_numpy(out[r]), ref, rtol=0, atol=1e-12), \
                "decode != torch SDPA"
            G = Hq // Hk
            sc = (qv @ K.repeat_interleave(G, 0).transpose(1, 2))[:, 0] * scale  # [Hq, n]
            ref_lse = torch.logsumexp(sc, dim=-1)
            assert torch.allclose(torch.from_numpy(lse[r]), ref_lse, rtol=0, atol=1e-12), \
                "decode lse != torch logsumexp"


def pin_permutation_invariance(orc):
    g = torch.Generator().manual_seed(17)
    q, pk, pv, pt, seq = _random_decode(g)
    R = pk.shape[0]
    perm = torch.randperm(R, generator=g)
    pk2, pv2 = torch.empty_like(pk), torch.empty_like(pv)
    pk2[perm] = pk
    pv2[perm] = pv
    pt2 = perm[pt.long()].to(torch.int32)
    a, la = orc.decode(q, pk, pv, pt, seq, 0.25)
    b, lb = orc.decode(q, pk2, pv2, pt2, seq, 0.25)
    assert np.array_equal(a, b) and np.array_equal(la, lb), "row relabelling changed the output"


def pin_page_size_equivalence(orc):
    """One request's logical K/V placed through single-row entries and through
    64-row pages (entries still raw rows) gives identical results."""
    g = torch.Generator().manual_seed(18)
    Hq, Hk, d, n, s = 4, 2, 16, 150, 64
    Kl, Vl = rnd((n, Hk, d), g), rnd((n, Hk, d), g)
    q = rnd((1, Hq, d), g)
    W = 160
    # page_size 1: rows scattered one by one
    R1 = 400
    rows1 = torch.randperm(R1, generator=g)[:n]
    pk1, pv1 = torch.zeros((R1, Hk, d), dtype=torch.bfloat16), torch.zeros((R1, Hk, d), dtype=torch.bfloat16)
    pk1[rows1], pv1[rows1] = Kl, Vl
    pt1 = torch.zeros((1, W), dtype=torch.int32)
    pt1[0, :n] = rows1.to(torch.int32)
    # page_size 64: whole pages at random page numbers
    npages_pool = 8
    pages = torch.randperm(npages_pool, generator=g)[: -(-n // s)]
    j = torch.arange(n)
    rows64 = pages[j // s] * s + j % s
    pk2 = torch.zeros((npages_pool * s, Hk, d), dtype=torch.bfloat16)
    pv2 = torch.zeros_like(pk2)
    pk2[rows64], pv2[rows64] = Kl, Vl
    pt2 = torch.zeros((1, W), dtype=torch.int32)
    pt2[0, :n] = rows64.to(torch.int32)
    seq = torch.tensor([n], dtype=torch.int32)
    a, la = orc.decode(q, pk1, pv1, pt1, seq, 0.25)
    b, lb = orc.decode(q, pk2, pv2, pt2, seq, 0.25)
    assert np.array_equal(a, b) and np.array_equal(la, lb), "page_size 1 vs 64 differ"


def pin_lse_merge(orc):
    g = torch.Generator().manual_seed(19)
    q, pk, pv, pt, seq = _random_decode(g, n_lo=9)
    full, full_lse = orc.decode(q, pk, pv, pt, seq, 0.3)
    B = q.shape[0]
    # three disjoint ranges covering [0, n), the middle one empty for request 0
    third = seq // 3
    cuts = [(torch.zeros(B, dtype=torch.int32), third), (third, third), (third, seq)]
    parts, lses = [], []
    for jb, je in cuts:
        o, l = orc.decode(q, pk, pv, pt, je.to(torch.int32), 0.3, j_begin=jb.to(torch.int32))
        parts.append(o)
        lses.append(l)
    assert np.all(np.isneginf(lses[1])), "empty range must have lse = -inf"
    mo, ml = orc.lse_merge(np.stack(parts), np.stack(lses))
    assert np.abs(mo - full).max() <= 1e-13, "merged partials != full softmax"
    assert np.abs(ml - full_lse).max() <= 1e-12, "merged lse != full lse"
    zo, zl = orc.lse_merge(np.stack([parts[1], parts[1]]), np.stack([lses[1], lses[1]]))
    assert np.all(zo == 0) and np.all(np.isneginf(zl)), "all-empty merge must give 0 / -inf"


def pin_poison_visible(orc):
    g = torch.Generator().manual_seed(20)
    q, pk, pv, pt, seq = _random_decode(g, n_hi=20)
    out, _ = orc.decode(q, pk, pv, pt, seq + 1, 0.3)  # one padding column read
    assert np.all(np.isnan(out)), "a NaN row read did not surface as NaN"


# --------------------------------------------------------------------------- #
# extend
# --------------------------------------------------------------------------- #
def _random_extend(g, cached, ext, Hq=8, Hk=2, d=16, R=None):
    B = len(cached)
    lens = [c + e for c, e in zip(cached, ext)]
    R = R or sum(lens) + 8
    pk, pv = rnd((R, Hk, d), g), rnd((R, Hk, d), g)
    pk[R - 1] = float("nan")
    pv[R - 1] = float("nan")
    W = ((max(lens) + 31) // 32) * 32
    pt = torch.full((B, W), R - 1, dtype=torch.int32)
    perm = torch.randperm(R - 1, generator=g)
    off = 0
    for r, n in enumerate(lens):
        pt[r, :n] = perm[off:off + n].to(torch.int32)
        off += n
    q = rnd((sum(ext), Hq, d), g)
    return q, pk, pv, pt, torch.tensor(cached, dtype=torch.int32), torch.tensor(ext, dtype=torch.int32)


def pin_extend_no_prefix_is_causal_sdpa(orc):
    g = torch.Generator().manual_seed(21)
    cached, ext = [0, 0, 0], [7, 1, 19]
    q, pk, pv, pt, cl, el = _random_extend(g, cached, ext)
    out = orc.extend(q, pk, pv, pt, cl, el, 0.3)
    off = 0
    for r, e in enumerate(ext):
        rows = pt[r, :e].long()
        K, V = f64(pk[rows]).permute(1, 0, 2), f64(pv[rows]).permute(1, 0, 2)
        qv = f64(q[off:off + e]).permute(1, 0, 2)
        ref = _sdpa(qv, K, V, 0.3, causal=True).permute(1, 0, 2)
        assert torch.allclose(torch.from_numpy(out[off:off + e]), ref, rtol=0, atol=1e-12), \
            "extend without prefix != causal SDPA"
        off += e


def pin_extend_with_prefix_masked_sdpa(orc):
    """New token t of a request with c cached tokens sees logical 0..c+t:
    a boolean mask aligned at the bottom-right corner."""
    g = torch.Generator().manual_seed(22)
    cached, ext = [5, 17, 0, 30], [9, 1, 4, 12]
    q, pk, pv, pt, cl, el = _random_extend(g, cached, ext)
    out = orc.extend(q, pk, pv, pt, cl, el, 0.3)
    off = 0
    for r, (c, e) in enumerate(zip(cached, ext)):
        n = c + e
        rows = pt[r, :n].long()
        K, V = f64(pk[rows]).permute(1, 0, 2), f64(pv[rows]).permute(1, 0, 2)
        qv = f64(q[off:off + e]).permute(1, 0, 2)
        mask = torch.ones((e, n), dtype=torch.bool).tril(diagonal=c)
        ref = _sdpa(qv, K, V, 0.3, mask=mask).permute(1, 0, 2)
        assert torch.allclose(torch.from_numpy(out[off:off + e]), ref, rtol=0, atol=1e-12), \
            "extend with prefix != bottom-right masked SDPA"
        off += e


def pin_extend_rows_equal_decode(orc):
    """Autoregressive consistency: extend's token t equals a decode of the same
    query over the first c+t+1 tokens."""
    g = torch.Generator().manual_seed(23)
    cached, ext = [11, 3], [6, 9]
    q, pk, pv, pt, cl, el = _random_extend(g, cached, ext)
    out = orc.extend(q, pk, pv, pt, cl, el, 0.3)
    off = 0
    for r, (c, e) in enumerate(zip(cached, ext)):
        for t in range(e):
            o, _ = orc.decode(q[off + t:off + t + 1], pk, pv, pt[r:r + 1],
                              torch.tensor([c + t + 1], dtype=torch.int32), 0.3)
            assert np.array_equal(o[0], out[off + t]), "extend row != decode over its prefix"
        off += e


def pin_extend_prefix_sharing(orc):
    """Requests that point at the same radix-cache prefix rows give exactly the
    results of requests that each hold a private copy of those rows."""
    g = torch.Generator().manual_seed(24)
    Hq, Hk, d, P = 8, 2, 16, 23
    ext = [5, 8, 3]
    B = len(ext)
    R = P * (B + 1) + sum(ext) + 4
    pk, pv = rnd((R, Hk, d), g), rnd((R, Hk, d), g)
    perm = torch.randperm(R, generator=g)
    shared = perm[:P]
    private = [perm[P * (i + 1):P * (i + 2)] for i in range(B)]
    off = P * (B + 1)
    own = []
    for e in ext:
        own.append(perm[off:off + e])
        off += e
    for p in private:
        pk[p], pv[p] = pk[shared], pv[shared]
    W = 32
    pt_s = torch.zeros((B, W), dtype=torch.int32)
    pt_p = torch.zeros((B, W), dtype=torch.int32)
    for r in range(B):
        pt_s[r, :P + ext[r]] = torch.cat([shared, own[r]]).to(torch.int32)
        pt_p[r, :P + ext[r]] = torch.cat([private[r], own[r]]).to(torch.int32)
    q = rnd((sum(ext), Hq, d), g)
    cl = torch.full((B,), P, dtype=torch.int32)
    el = torch.tensor(ext, dtype=torch.int32)
    a = orc.extend(q, pk, pv, pt_s, cl, el, 0.3)
    b = orc.extend(q, pk, pv, pt_p, cl, el, 0.3)
    assert np.array_equal(a, b), "shared prefix rows != private copies"


# --------------------------------------------------------------------------- #
# CUDA-Graph padding requests
# --------------------------------------------------------------------------- #
def pin_dummy_requests(orc):
    """Padding requests point every page-table entry and their out_loc at the
    dummy row; their stores and reads never touch a real row, and their output
    is V of the dummy row."""
    g = torch.Generator().manual_seed(25)
    Hq, Hk, d, R = 8, 2, 16, 128
    n_real, n_dummy = 3, 4
    D = R - 2
    pk, pv = rnd((R, Hk, d), g), rnd((R, Hk, d), g)
    B = n_real + n_dummy
    W = 32
    pt = torch.full((B, W), D, dtype=torch.int32)
    perm = torch.randperm(D, generator=g)
    seq = torch.tensor([9, 4, 13] + [1, 1, 28, 5], dtype=torch.int32)  # padding: any length <= W
    off = 0
    for r in range(n_real):
        n = int(seq[r])
        pt[r, :n] = perm[off:off + n].to(torch.int32)
        off += n
    loc = torch.tensor([int(pt[r, int(seq[r]) - 1]) for r in range(B)], dtype=torch.int32)
    k_new, v_new = rnd((B, Hk, d), g), rnd((B, Hk, d), g)
    k_new[n_real:] = k_new[n_real]
    v_new[n_real:] = v_new[n_real]
    ok, ov = u16(pk), u16(pv)
    before_k, before_v = ok.copy(), ov.copy()
    orc.store_kv(ok, ov, k_new, v_new, loc)
    touched = set(loc[:n_real].tolist()) | {D}
    for row in range(R):
        if row not in touched:
            assert np.array_equal(ok[row], before_k[row]) and np.array_equal(ov[row], before_v[row]), \
                "a row outside out_loc changed"
    assert np.array_equal(ov[D], u16(v_new[n_real])), "dummy row does not hold the padding value"
    q = rnd((B, Hq, d), g)
    out, _ = orc.decode(q, ok.reshape(R, Hk, d), ov.reshape(R, Hk, d), pt, seq, 0.3)
    vd = f64(v_new[n_real]).numpy()
    G = Hq // Hk
    for r in range(n_real, B):
        for h in range(Hq):
            assert np.array_equal(out[r, h], vd[h // G]), "padding request output != V[dummy]"


# --------------------------------------------------------------------------- #
# golden fixtures
# --------------------------------------------------------------------------- #
def pin_golden_page_table_example(orc):
    with open(os.path.join(GOLDEN, "page_table_example.json")) as f:
        fx = json.load(f)
    d = fx["head_dim"]
    K = np.array(fx["K"], dtype=np.float64)
    V = np.array(fx["V"], dtype=np.float64)
    R = K.shape[0]
    pk = bf16(K).reshape(R, 1, d)
    pv = bf16(V).reshape(R, 1, d)
    assert torch.equal(f64(pk).reshape(R, d), torch.from_numpy(K)), "fixture values must be bf16-exact"
    tables = fx["page_table"]
    W = 32
    pt = torch.zeros((len(tables), W), dtype=torch.int32)
    for r, rows in enumerate(tables):
        pt[r, :len(rows)] = torch.tensor(rows, dtype=torch.int32)
    seq = torch.tensor([len(t) for t in tables], dtype=torch.int32)
    q = bf16(np.array(fx["q"], dtype=np.float64)).reshape(len(tables), 1, d)
    scale = eval(fx["sm_scale"], {"__builtins__": {}}, {"log": math.log})
    out, lse = orc.decode(q, pk, pv, pt, seq, scale)
    ev = lambda e: float(eval(e, {"__builtins__": {}}, {"log": math.log, "sqrt": math.sqrt}))
    exp_o = np.array([[ev(e) for e in row] for row in fx["expected_out"]], dtype=np.float64)
    exp_l = np.array([ev(e) for e in fx["expected_lse"]], dtype=np.float64)
    assert np.abs(out[:, 0] - exp_o).max() <= 1e-12, "golden page-table example: output"
    assert np.abs(lse[:, 0] - exp_l).max() <= 1e-12, "golden page-table example: lse"


# --------------------------------------------------------------------------- #
# rotary position embedding (deep dive, section 7.3)
# --------------------------------------------------------------------------- #
def _angles(d, positions, base=10000.0):
    """theta[p, i] = p * base^(-2i/d) in float64 (the pages' frequencies)."""
    inv = base ** (-np.arange(0, d, 2, dtype=np.float64) / d)
    return np.outer(np.asarray(positions, dtype=np.float64), inv)


def _cos_sin_table(d, max_pos, base=10000.0):
    """[cos | sin] rows per position, float32 as the pages store them."""
    ang = _angles(d, np.arange(max_pos), base)
    return np.concatenate([np.cos(ang), np.sin(ang)], 1).astype(np.float32)


def pin_rope_position_zero_is_identity(orc):
    g = torch.Generator().manual_seed(31)
    x = rnd((5, 3, 16), g)
    out = orc.rope(x, np.zeros(5, dtype=np.int32), _cos_sin_table(16, 8))
    assert np.array_equal(out, f64(x).numpy()), "position 0 must leave x unchanged"


def pin_rope_is_complex_rotation(orc):
    """RoPE multiplies z_i = x_i + 1j*x_{i+d/2} by exp(1j*theta_i); the
    reference uses numpy's complex exponential, not the cached table, so the
    tolerance covers the table's float32 rounding."""
    g = torch.Generator().manual_seed(32)
    N, H, d = 9, 3, 16
    x = rnd((N, H, d), g)
    pos = torch.randint(0, 60, (N,), generator=g).numpy().astype(np.int32)
    out = orc.rope(x, pos, _cos_sin_table(d, 64))
    xf = f64(x).numpy()
    z = xf[..., : d // 2] + 1j * xf[..., d // 2:]
    w = z * np.exp(1j * _angles(d, pos))[:, None, :]
    ref = np.concatenate([w.real, w.imag], -1)
    assert np.abs(out - ref).max() <= 1e-6 * (np.abs(xf).max() + 1.0), "not a rotation by +theta"


def pin_rope_relative_position(orc):
    """<R(p) q, R(p') k> depends on p - p' only (the property RoPE exists for)."""
    g = torch.Generator().manual_seed(33)
    d = 32
    q = rnd((1, 1, d), g)
    k = rnd((1, 1, d), g)
    table = _cos_sin_table(d, 256)
    one = lambda x, p: orc.rope(x, np.array([p], dtype=np.int32), table).reshape(d)
    scale = float(torch.linalg.norm(f64(q)) * torch.linalg.norm(f64(k)))
    for p, pp, delta in ((3, 10, 17), (40, 2, 100), (0, 0, 200), (7, 7, 1)):
        a = float(np.dot(one(q, p), one(k, pp)))
        b = float(np.dot(one(q, p + delta), one(k, pp + delta)))
        assert abs(a - b) <= 1e-5 * scale, ("relative position", p, pp, delta)
    # and it does depend on the offset
    assert abs(float(np.dot(one(q, 0), one(k, 0))) - float(np.dot(one(q, 0), one(k, 5)))) > 1e-3 * scale


def pin_rope_rejects_positions_outside_table(orc):
    x = rnd((2, 1, 8), torch.Generator().manual_seed(34))
    for bad in ([0, 4], [-1, 0]):
        try:
            orc.rope(x, np.array(bad, dtype=np.int32), _cos_sin_table(8, 4))
        except ValueError:
            continue
        raise AssertionError("a position outside the table was accepted")


ALL_PINS = [
    pin_store_kv_index_put,
    pin_single_token_returns_v,
    pin_equal_scores_mean,
    pin_decode_matches_sdpa,
    pin_permutation_invariance,
    pin_page_size_equivalence,
    pin_lse_merge,
    pin_poison_visible,
    pin_extend_no_prefix_is_causal_sdpa,
    pin_extend_with_prefix_masked_sdpa,
    pin_extend_rows_equal_decode,
    pin_extend_prefix_sharing,
    pin_dummy_requests,
    pin_golden_page_table_example,
    pin_rope_position_zero_is_identity,
    pin_rope_is_complex_rotation,
    pin_rope_relative_position,
    pin_rope_rejects_positions_outside_table,
]
