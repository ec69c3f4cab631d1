"""Seeded synthetic inputs for paged KV-pool attention.

This module draws the inputs only: context lengths, where each token's K/V row
sits in the pool, the page tables and out_loc vectors that point at those rows,
and the K/V/Q values.  It holds none of the attention arithmetic.  The oracle
tests, the GPU parity tests and bench.py all take their inputs from here, so
both sides of every comparison see the same numbers.

Vocabulary follows the mini-sglang pages:
  * pool: one tensor per layer stack, logical shape (2, L, R, H_kv, d), K then V,
    LayerFirst ("mini-sglang architecture deep dive", section 6.2 MHAKVCache);
    per layer K and V are each an (R, H_kv, d) array of token rows whose
    physical position is the row number (mini-sglang-learn, paged KV pool).
  * page_table[r, j]: the physical row of logical token j of request r; raw
    rows, not page numbers; width padded up to a multiple of 32
    (mini-sglang-learn, page_table alignment passage).
  * out_loc[i]: the row where token i's new K/V go (mini-sglang-learn,
    store_kv passage).
  * one extra dummy row, pointed at by every entry of a CUDA-Graph padding
    request (mini-sglang-learn, dummy page passage).

Two rows are reserved past the live rows: DUMMY (R-2) and POISON (R-1).  The
poison row holds NaN in every layer and fills the page_table past each
request's length, so any read of a padding column shows up as NaN.

Generation order within a case follows one fixed recipe: lengths, row
permutation, page_table, out_loc; values (pool, new k/v, q) come after, from a
second generator seeded from the same seed, so the index structure of a case
does not depend on the device its values are drawn on.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

ALIGN = 32


def align_up(x: int, a: int = ALIGN) -> int:
    return ((x + a - 1) // a) * a


# --------------------------------------------------------------------------- #
# decode cases
# --------------------------------------------------------------------------- #
@dataclass
class DecodeCase:
    name: str
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    batch: int              # requests including CUDA-Graph padding requests
    num_real: int           # the first num_real requests are real
    num_rows: int           # R: rows per layer, including the dummy and poison rows
    seq_lens: torch.Tensor  # [B] int32, context length incl. the token stored this step
    page_table: torch.Tensor  # [B, W] int32
    out_loc: torch.Tensor   # [B] int32, row of the token stored this step
    sm_scale: float
    value_std: float
    seed: int

    @property
    def dummy_row(self) -> int:
        return self.num_rows - 2

    @property
    def poison_row(self) -> int:
        return self.num_rows - 1

    @property
    def width(self) -> int:
        return int(self.page_table.shape[1])


def _real_rows_needed(lengths: List[int], page_size: int) -> int:
    if page_size == 1:
        return sum(lengths)
    return sum(-(-n // page_size) for n in lengths) * page_size


def make_decode_case(name: str, *, num_layers: int, num_q_heads: int, num_kv_heads: int,
                     head_dim: int, page_size: int, batch: int, ctx_lo: int, ctx_hi: int,
                     ctx_dist: str = "uniform", num_dummy: int = 0, dummy_seq_len: int = 1,
                     pool_factor: float = 1.2, min_rows: int = 0, value_std: float = 1.0,
                     seed: int = 0) -> DecodeCase:
    """Draw the index structure of one decode step.

    ctx is the cached context before this step; the step stores one new token
    per request, so seq_len = ctx + 1 and the new row is page_table[r, ctx].
    Real requests take their rows from a random permutation of the pool
    (page_size 1) or from whole pages at random page indices (page_size > 1).
    Padding requests (num_dummy of them, at the end of the batch) point every
    page_table entry and their out_loc at the dummy row.
    """
    g = torch.Generator().manual_seed(seed)
    n_real = batch - num_dummy
    # 1. lengths
    if ctx_dist == "uniform":
        ctx = torch.randint(ctx_lo, ctx_hi + 1, (n_real,), generator=g)
    elif ctx_dist == "loguniform":
        u = torch.rand((n_real,), generator=g, dtype=torch.float64)
        ctx = torch.exp(math.log(ctx_lo) + u * (math.log(ctx_hi) - math.log(ctx_lo)))
        ctx = ctx.round().clamp(ctx_lo, ctx_hi).to(torch.int64)
    else:
        raise ValueError(ctx_dist)
    seq = [int(c) + 1 for c in ctx.tolist()]
    # 2. row permutation
    need = _real_rows_needed(seq, page_size)
    live = max(int(math.ceil(pool_factor * need)), min_rows, need)
    if page_size > 1:
        live = align_up(live, page_size)
    R = live + 2
    dummy, poison = R - 2, R - 1
    width = align_up(max(seq + [dummy_seq_len if num_dummy else 1]))
    pt = torch.full((batch, width), poison, dtype=torch.int32)
    if page_size == 1:
        perm = torch.randperm(live, generator=g).to(torch.int32)
        off = 0
        for r, n in enumerate(seq):
            pt[r, :n] = perm[off:off + n]
            off += n
    else:
        pages = torch.randperm(live // page_size, generator=g)
        off = 0
        for r, n in enumerate(seq):
            npg = -(-n // page_size)
            mine = pages[off:off + npg]
            off += npg
            j = torch.arange(n)
            pt[r, :n] = (mine[j // page_size] * page_size + j % page_size).to(torch.int32)
    # 3. padding requests
    for r in range(n_real, batch):
        pt[r, :] = dummy
    seq_lens = torch.tensor(seq + [dummy_seq_len] * num_dummy, dtype=torch.int32)
    # 4. out_loc: the row holding logical token seq_len-1
    out_loc = torch.empty(batch, dtype=torch.int32)
    for r in range(batch):
        out_loc[r] = pt[r, int(seq_lens[r]) - 1]
    return DecodeCase(name=name, num_layers=num_layers, num_q_heads=num_q_heads,
                      num_kv_heads=num_kv_heads, head_dim=head_dim, page_size=page_size,
                      batch=batch, num_real=n_real, num_rows=R, seq_lens=seq_lens,
                      page_table=pt, out_loc=out_loc, sm_scale=1.0 / math.sqrt(head_dim),
                      value_std=value_std, seed=seed)


# The five workloads, by what they are.
def decode_tiny(seed: int = 1000) -> DecodeCase:
    """Batch 4, H_q 8, H_kv 2, d 64, one layer, page_size 1, 4096-row pool, N(0,1)."""
    return make_decode_case("tiny-decode-b4-gqa4-d64", num_layers=1, num_q_heads=8,
                            num_kv_heads=2, head_dim=64, page_size=1, batch=4, ctx_lo=16,
                            ctx_hi=128, min_rows=4096, pool_factor=1.0, value_std=1.0,
                            seed=seed)


def decode_qwen3_0p6b(seed: int = 1001, num_layers: int = 28,
                      pool_factor: float = 1.2) -> DecodeCase:
    """Qwen3-0.6B attention shapes: 28 layers, H_q 16, H_kv 8, d 128, batch 64, ctx U[512,4096]."""
    return make_decode_case("qwen3-0.6b-decode-b64-ctx512-4096", num_layers=num_layers,
                            num_q_heads=16, num_kv_heads=8, head_dim=128, page_size=1,
                            batch=64, ctx_lo=512, ctx_hi=4096, value_std=0.5,
                            pool_factor=pool_factor, seed=seed)


def decode_llama3_8b(seed: int = 1002, num_layers: int = 32,
                     pool_factor: float = 1.2) -> DecodeCase:
    """Llama-3-8B attention shapes: 32 layers, H_q 32, H_kv 8, d 128; 200 real requests
    with log-uniform ctx in [1024,8192], padded with 56 dummy requests to batch 256.
    The pool holds pool_factor times the live tokens (1.2; 1.05 where memory is short)."""
    return make_decode_case("llama3-8b-decode-b200pad256-ctx1k-8k", num_layers=num_layers,
                            num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=1,
                            batch=256, num_dummy=56, ctx_lo=1024, ctx_hi=8192,
                            ctx_dist="loguniform", value_std=0.5, pool_factor=pool_factor,
                            seed=seed)


def decode_pool_bytes(case: DecodeCase) -> int:
    """Bytes of the (2, L, R, H_kv, d) bf16 pool of a decode case."""
    return 2 * case.num_layers * case.num_rows * case.num_kv_heads * case.head_dim * 2


def decode_long_page64(seed: int = 1004) -> DecodeCase:
    """Long context with 64-row pages: H_q 64, H_kv 8, d 128, batch 32, ctx U[8192,32768]."""
    return make_decode_case("long-decode-page64-b32-ctx8k-32k", num_layers=1, num_q_heads=64,
                            num_kv_heads=8, head_dim=128, page_size=64, batch=32,
                            ctx_lo=8192, ctx_hi=32768, value_std=0.5, seed=seed)


# --------------------------------------------------------------------------- #
# extend (chunked prefill) cases
# --------------------------------------------------------------------------- #
@dataclass
class ExtendBatch:
    req_ids: List[int]
    cached_lens: torch.Tensor   # [B] int32
    extend_lens: torch.Tensor   # [B] int32
    q_offsets: torch.Tensor     # [B+1] int32, exclusive prefix sum of extend_lens
    page_table: torch.Tensor    # [B, W] int32
    out_loc: torch.Tensor       # [T] int32, the new rows in request order

    @property
    def total_tokens(self) -> int:
        return int(self.q_offsets[-1])


@dataclass
class ExtendCase:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    num_rows: int
    prefix_rows: torch.Tensor   # [prefix_len] int32, shared by every request
    extend_lens: List[int]      # full extend length of each request
    batches: List[ExtendBatch] = field(default_factory=list)
    sm_scale: float = 0.0
    value_std: float = 0.5
    seed: int = 0
    num_layers: int = 1

    @property
    def poison_row(self) -> int:
        return self.num_rows - 1

    @property
    def dummy_row(self) -> int:
        return self.num_rows - 2


def make_extend_case(name: str, *, num_q_heads: int, num_kv_heads: int, head_dim: int,
                     num_reqs: int, prefix_len: int, ext_lo: int, ext_hi: int, budget: int,
                     pool_factor: float = 1.2, value_std: float = 0.5, seed: int = 0,
                     shared_prefix: bool = True) -> ExtendCase:
    """Draw requests that share one cached prefix and then add ext ~ U[ext_lo, ext_hi]
    new tokens each, and cut them into batches of at most `budget` new tokens.

    Batching takes requests in order; each gets chunk = min(budget left, tokens
    it still has to extend).  A request cut short continues at the head of the
    next batch with cached_len = prefix_len + tokens already done, and the rows
    of its earlier chunks already sit in its page_table row
    (mini-sglang-learn, chunked prefill passage: chunk_size = min(budget,
    remaining), the chunked request keeps its table slot).
    With shared_prefix=False every request gets a private copy of the prefix
    rows (different physical rows, same values are the caller's business).
    """
    g = torch.Generator().manual_seed(seed)
    ext = torch.randint(ext_lo, ext_hi + 1, (num_reqs,), generator=g).tolist()
    n_prefix_copies = 1 if shared_prefix else num_reqs
    need = prefix_len * n_prefix_copies + sum(ext)
    live = int(math.ceil(pool_factor * need))
    R = live + 2
    perm = torch.randperm(live, generator=g).to(torch.int32)
    off = 0
    prefix_of = []
    for i in range(n_prefix_copies):
        prefix_of.append(perm[off:off + prefix_len].clone())
        off += prefix_len
    if shared_prefix:
        prefix_of = prefix_of * num_reqs
    new_rows = []
    for e in ext:
        new_rows.append(perm[off:off + e].clone())
        off += e
    case = ExtendCase(name=name, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                      head_dim=head_dim, num_rows=R, prefix_rows=prefix_of[0],
                      extend_lens=ext, sm_scale=1.0 / math.sqrt(head_dim),
                      value_std=value_std, seed=seed)
    case.prefix_rows_per_req = prefix_of  # type: ignore[attr-defined]
    done = [0] * num_reqs
    r = 0
    while r < num_reqs:
        left = budget
        ids, cl, el = [], [], []
        while r < num_reqs and left > 0:
            chunk = min(left, ext[r] - done[r])
            ids.append(r)
            cl.append(prefix_len + done[r])
            el.append(chunk)
            left -= chunk
            done[r] += chunk
            if done[r] == ext[r]:
                r += 1
            else:
                break  # cut short: continues first in the next batch
        lens = [c + e for c, e in zip(cl, el)]
        width = align_up(max(lens))
        pt = torch.full((len(ids), width), R - 1, dtype=torch.int32)
        outs = []
        for b, (rid, c, e) in enumerate(zip(ids, cl, el)):
            pt[b, :prefix_len] = prefix_of[rid]
            own = new_rows[rid][: c + e - prefix_len]
            pt[b, prefix_len:c + e] = own
            outs.append(own[c - prefix_len:])
        qo = torch.zeros(len(ids) + 1, dtype=torch.int32)
        qo[1:] = torch.cumsum(torch.tensor(el, dtype=torch.int32), 0)
        case.batches.append(ExtendBatch(req_ids=ids, cached_lens=torch.tensor(cl, dtype=torch.int32),
                                        extend_lens=torch.tensor(el, dtype=torch.int32),
                                        q_offsets=qo.to(torch.int32), page_table=pt,
                                        out_loc=torch.cat(outs).to(torch.int32)))
    return case


def extend_radix_shared(seed: int = 1003) -> ExtendCase:
    """32 requests sharing a 2048-token cached prefix (same physical rows), each adding
    U[256,1024] new tokens, batched at 8192 new tokens; H_q 32, H_kv 8, d 128."""
    return make_extend_case("radix-shared-extend-32req-prefix2048", num_q_heads=32,
                            num_kv_heads=8, head_dim=128, num_reqs=32, prefix_len=2048,
                            ext_lo=256, ext_hi=1024, budget=8192, value_std=0.5, seed=seed)


# --------------------------------------------------------------------------- #
# values
# --------------------------------------------------------------------------- #
def _normal_(t: torch.Tensor, std: float, g: torch.Generator) -> torch.Tensor:
    return t.normal_(0.0, std, generator=g)


def make_pool(num_layers: int, num_rows: int, num_kv_heads: int, head_dim: int, std: float,
              seed: int, device: str = "cpu") -> torch.Tensor:
    """(2, L, R, H_kv, d) bf16 pool with N(0, std^2) values, drawn layer by layer on
    `device`; the last row of every layer (the poison row) is NaN."""
    g = torch.Generator(device=device).manual_seed(seed * 7919 + 17)
    pool = torch.empty((2, num_layers, num_rows, num_kv_heads, head_dim), dtype=torch.bfloat16,
                       device=device)
    for kv in range(2):
        for layer in range(num_layers):
            _normal_(pool[kv, layer], std, g)
    pool[:, :, num_rows - 1] = float("nan")
    return pool


def make_decode_values(case: DecodeCase, device: str = "cpu"):
    """Pool, new k/v [L, B, H_kv, d] and q [L, B, H_q, d] for a decode case.

    Padding requests all store the same k/v values (one fixed random row), so
    their racing writes to the dummy row agree byte for byte."""
    pool = make_pool(case.num_layers, case.num_rows, case.num_kv_heads, case.head_dim,
                     case.value_std, case.seed, device)
    g = torch.Generator(device=device).manual_seed(case.seed * 104729 + 3)
    L, B, Hk, Hq, d = case.num_layers, case.batch, case.num_kv_heads, case.num_q_heads, case.head_dim
    k_new = _normal_(torch.empty((L, B, Hk, d), dtype=torch.bfloat16, device=device), case.value_std, g)
    v_new = _normal_(torch.empty((L, B, Hk, d), dtype=torch.bfloat16, device=device), case.value_std, g)
    if case.num_real < B:
        k_new[:, case.num_real:] = k_new[:, case.num_real:case.num_real + 1].clone()
        v_new[:, case.num_real:] = v_new[:, case.num_real:case.num_real + 1].clone()
    q = _normal_(torch.empty((L, B, Hq, d), dtype=torch.bfloat16, device=device), case.value_std, g)
    return pool, k_new, v_new, q


def make_extend_values(case: ExtendCase, device: str = "cpu"):
    """Pool (one layer) plus, per batch, new k/v [T, H_kv, d] and q [T, H_q, d]."""
    pool = make_pool(case.num_layers, case.num_rows, case.num_kv_heads, case.head_dim,
                     case.value_std, case.seed, device)
    g = torch.Generator(device=device).manual_seed(case.seed * 104729 + 5)
    per_batch = []
    for b in case.batches:
        T = b.total_tokens
        k = _normal_(torch.empty((T, case.num_kv_heads, case.head_dim), dtype=torch.bfloat16,
                                 device=device), case.value_std, g)
        v = _normal_(torch.empty((T, case.num_kv_heads, case.head_dim), dtype=torch.bfloat16,
                                 device=device), case.value_std, g)
        q = _normal_(torch.empty((T, case.num_q_heads, case.head_dim), dtype=torch.bfloat16,
                                 device=device), case.value_std, g)
        per_batch.append((k, v, q))
    return pool, per_batch


# --------------------------------------------------------------------------- #
# rotary position embedding inputs
# --------------------------------------------------------------------------- #
def rope_cos_sin_cache(head_dim: int, max_positions: int, base: float = 10000.0) -> torch.Tensor:
    """The cos/sin table a serving engine builds once at start-up for RoPE
    ("mini-sglang architecture deep dive", section 7.3): row p holds
    [cos(p f_0) .. cos(p f_{d/2-1}), sin(p f_0) .. sin(p f_{d/2-1})] with
    f_i = base^(-2i/d), in float32 (rotary_dim = head_dim).  It is an input to
    the RoPE step, like the pool; the pages give no base, 10000 is used."""
    freq = 1.0 / (base ** (torch.arange(0, head_dim, 2, dtype=torch.float32) / head_dim))
    ang = torch.outer(torch.arange(max_positions, dtype=torch.float32), freq)
    return torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).contiguous()


def decode_positions(case: DecodeCase) -> torch.Tensor:
    """Position of the token each request stores this step: its context
    length minus one (the context includes that token).  Padding requests
    all use position 0, so their rotated keys agree byte for byte."""
    pos = (case.seq_lens - 1).clamp(min=0).to(torch.int32)
    if case.num_real < case.batch:
        pos[case.num_real:] = 0
    return pos


def extend_positions(batch: ExtendBatch) -> torch.Tensor:
    """Positions of the packed new tokens of an extend batch: request r's new
    token t sits at cached_len[r] + t."""
    parts = [torch.arange(int(c), int(c) + int(e), dtype=torch.int32)
             for c, e in zip(batch.cached_lens.tolist(), batch.extend_lens.tolist())]
    return torch.cat(parts) if parts else torch.zeros(0, dtype=torch.int32)


# --------------------------------------------------------------------------- #
# decode with a radix-shared prefix
# --------------------------------------------------------------------------- #
def make_shared_prefix_decode_case(name: str, *, num_q_heads: int, num_kv_heads: int,
                                   head_dim: int, batch: int, prefix_len: int, suffix_lo: int,
                                   suffix_hi: int, pool_factor: float = 1.2,
                                   value_std: float = 0.5, seed: int = 0) -> DecodeCase:
    """Decode step for requests that all matched one cached prefix: the first
    prefix_len page-table entries of every request are the same physical rows
    (mini-sglang-learn, radix-cache chapter), followed by a private suffix of
    U[suffix_lo, suffix_hi] cached tokens and the token stored this step.
    Rows come from one random permutation of the pool; one layer."""
    g = torch.Generator().manual_seed(seed)
    suf = torch.randint(suffix_lo, suffix_hi + 1, (batch,), generator=g).tolist()
    seq = [prefix_len + s + 1 for s in suf]
    need = prefix_len + sum(s + 1 for s in suf)
    live = max(int(math.ceil(pool_factor * need)), need)
    R = live + 2
    poison = R - 1
    perm = torch.randperm(live, generator=g).to(torch.int32)
    width = align_up(max(seq))
    pt = torch.full((batch, width), poison, dtype=torch.int32)
    pt[:, :prefix_len] = perm[:prefix_len]
    off = prefix_len
    for r, n in enumerate(seq):
        k = n - prefix_len
        pt[r, prefix_len:n] = perm[off:off + k]
        off += k
    seq_lens = torch.tensor(seq, dtype=torch.int32)
    out_loc = torch.tensor([int(pt[r, n - 1]) for r, n in enumerate(seq)], dtype=torch.int32)
    case = DecodeCase(name=name, num_layers=1, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                      head_dim=head_dim, page_size=1, batch=batch, num_real=batch, num_rows=R,
                      seq_lens=seq_lens, page_table=pt, out_loc=out_loc,
                      sm_scale=1.0 / math.sqrt(head_dim), value_std=value_std, seed=seed)
    case.shared_len = prefix_len  # type: ignore[attr-defined]
    return case


def decode_shared_prefix_qwen3(seed: int = 1005, prefix_len: int = 4096) -> DecodeCase:
    """Qwen3-0.6B-shaped decode (H_q 16, H_kv 8, d 128) for 64 requests that
    share a cached prefix (4096 tokens by default) and add private suffixes
    of U[16, 512]."""
    return make_shared_prefix_decode_case(f"shared-prefix-decode-b64-p{prefix_len}-s16-512",
                                          num_q_heads=16, num_kv_heads=8, head_dim=128, batch=64,
                                          prefix_len=prefix_len, suffix_lo=16, suffix_hi=512,
                                          seed=seed)


# --------------------------------------------------------------------------- #
# a mixed batch: chunked prefill and decode requests in one extend call
# --------------------------------------------------------------------------- #
def mixed_chunk_decode(seed: int = 1006, num_decode: int = 64, ctx_lo: int = 512,
                       ctx_hi: int = 4096) -> ExtendCase:
    """One mixed batch as SGLang's mixed-chunk mode forms it ("SGLang 源码导读",
    --enable-mixed-chunk): the first chunked-prefill batch of the radix-shared
    extend workload (requests sharing a 2048-token prefix, up to 8192 new
    tokens) followed by `num_decode` decode requests, each adding one token
    over U[ctx_lo, ctx_hi] cached tokens (the Qwen3-0.6B decode context mix);
    H_q 32, H_kv 8, d 128.  Returns a one-batch ExtendCase; the decode
    requests are the last `num_decode` of the batch (case.num_decode)."""
    base = extend_radix_shared()
    b0 = base.batches[0]
    g = torch.Generator().manual_seed(seed)
    ctx = torch.randint(ctx_lo, ctx_hi + 1, (num_decode,), generator=g).tolist()
    live_base = base.num_rows - 2
    n_dec_rows = sum(c + 1 for c in ctx)
    R = live_base + n_dec_rows + 2
    poison = R - 1
    perm = (torch.randperm(n_dec_rows, generator=g) + live_base).to(torch.int32)
    lens = [int(c) + int(e) for c, e in zip(b0.cached_lens.tolist(), b0.extend_lens.tolist())]
    width = align_up(max(lens + [c + 1 for c in ctx]))
    nb = len(lens)
    pt = torch.full((nb + num_decode, width), poison, dtype=torch.int32)
    for r, n in enumerate(lens):
        pt[r, :n] = b0.page_table[r, :n]
    outs = [b0.out_loc]
    off = 0
    for i, c in enumerate(ctx):
        rows = perm[off:off + c + 1]
        off += c + 1
        pt[nb + i, :c + 1] = rows
        outs.append(rows[c:c + 1])
    cl = torch.cat([b0.cached_lens, torch.tensor(ctx, dtype=torch.int32)])
    el = torch.cat([b0.extend_lens, torch.ones(num_decode, dtype=torch.int32)])
    qo = torch.zeros(nb + num_decode + 1, dtype=torch.int32)
    qo[1:] = torch.cumsum(el, 0)
    case = ExtendCase(name=f"mixed-chunk8192-plus-{num_decode}-decode", num_q_heads=base.num_q_heads,
                      num_kv_heads=base.num_kv_heads, head_dim=base.head_dim, num_rows=R,
                      prefix_rows=base.prefix_rows, extend_lens=el.tolist(), sm_scale=base.sm_scale,
                      value_std=base.value_std, seed=seed)
    case.batches.append(ExtendBatch(req_ids=list(range(nb + num_decode)), cached_lens=cl.to(torch.int32),
                                    extend_lens=el.to(torch.int32), q_offsets=qo.to(torch.int32),
                                    page_table=pt, out_loc=torch.cat(outs).to(torch.int32)))
    case.num_decode = num_decode  # type: ignore[attr-defined]
    return case


# --------------------------------------------------------------------------- #
# store_kv at scale: several disjoint extend-sized batches
# --------------------------------------------------------------------------- #
@dataclass
class StoreRotation:
    name: str
    num_rows: int
    num_kv_heads: int
    head_dim: int
    out_locs: List[torch.Tensor]  # one [tokens] int32 per batch, rows disjoint across batches
    seed: int


def store_rotation(seed: int = 1007, batches: int = 8, tokens: int = 8192, num_kv_heads: int = 8,
                   head_dim: int = 128, pool_factor: float = 1.2) -> StoreRotation:
    """`batches` store_kv batches of `tokens` new tokens each (the chunked-prefill
    budget of the radix-shared extend workload), with disjoint random rows of
    one pool, so that storing them one after the other touches more memory than
    the L2 holds (8 x 67 MB at the defaults)."""
    g = torch.Generator().manual_seed(seed)
    live = int(math.ceil(pool_factor * batches * tokens))
    perm = torch.randperm(live, generator=g).to(torch.int32)
    locs = [perm[b * tokens:(b + 1) * tokens].clone() for b in range(batches)]
    return StoreRotation(name=f"store-kv-{batches}x{tokens}-tokens", num_rows=live + 2,
                         num_kv_heads=num_kv_heads, head_dim=head_dim, out_locs=locs, seed=seed)
