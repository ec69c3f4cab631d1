"""Helpers shared by the GPU parity tests (marshalling and comparisons only).

Oracle inputs are always the generator's values copied from the device BEFORE
any library kernel runs; new rows reach the oracle's copy of the pool through
the oracle's own store_kv, never through the CUDA path's output.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle

# attention tolerance against the fp64 oracle
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def check_attn(gpu: torch.Tensor, ref: np.ndarray, what: str) -> dict:
    g = gpu.detach().float().cpu().double().numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(ref).all(), f"{what}: oracle produced non-finite values"
    assert np.isfinite(g).all(), f"{what}: GPU output has non-finite values"
    err = np.abs(g - ref)
    stats = {"max_abs": float(err.max()), "mean_abs": float(err.mean())}
    assert stats["max_abs"] <= MAX_ABS and stats["mean_abs"] <= MEAN_ABS, f"{what}: {stats}"
    return stats


class CompactPool:
    """Host copy of just the pool rows some requests touch, with the page
    table rewritten to index the copy.  Rows are gathered from the device
    pool tensor (generator values) before any kernel writes to it."""

    def __init__(self, k_layer: torch.Tensor, v_layer: torch.Tensor, rows: torch.Tensor):
        self.rows = torch.unique(rows.to(torch.int64).cpu())  # sorted
        idx = self.rows.to(k_layer.device)
        self.k = u16(k_layer.index_select(0, idx))
        self.v = u16(v_layer.index_select(0, idx))

    def remap(self, phys: torch.Tensor) -> torch.Tensor:
        p = phys.to(torch.int64).cpu()
        pos = torch.searchsorted(self.rows, p)
        pos = pos.clamp(max=len(self.rows) - 1)
        assert torch.equal(self.rows[pos], p), "row outside the compact set"
        return pos.to(torch.int32)

    def store(self, k_new, v_new, out_loc) -> None:
        oracle.get().store_kv(self.k, self.v, k_new, v_new, self.remap(out_loc))


def request_rows(page_table: torch.Tensor, lens, reqs) -> torch.Tensor:
    return torch.cat([page_table[r, :int(lens[r])] for r in reqs])


def oracle_decode_requests(cp: CompactPool, q, page_table, seq_lens, reqs, sm_scale):
    """Oracle decode for a subset of requests on a compact pool."""
    W = page_table.shape[1]
    pt = torch.zeros((len(reqs), W), dtype=torch.int32)
    sl = torch.zeros(len(reqs), dtype=torch.int32)
    for i, r in enumerate(reqs):
        n = int(seq_lens[r])
        sl[i] = n
        if n:
            pt[i, :n] = cp.remap(page_table[r, :n])
    qs = q[list(reqs)].cpu()
    return oracle.get().decode(qs, cp.k, cp.v, pt, sl, sm_scale)


def host_threads() -> int:
    """Threads for the oracle: one per host core this process may run on."""
    return max(1, len(os.sched_getaffinity(0)))


def parallel_oracle_decode(k_host, v_host, q, page_table, seq_lens, sm_scale, reqs=None):
    """Oracle decode of requests `reqs` (all by default) over a whole host
    layer (uint16 [R, H_kv, d] arrays), requests dealt round-robin to one
    thread per host core.  Each thread calls the single-threaded C oracle on
    its own requests (ctypes releases the GIL), so the arithmetic is exactly
    the oracle's.  Returns out [len(reqs), H_q, d] float64 and lse."""
    orc = oracle.get()
    reqs = list(range(page_table.shape[0])) if reqs is None else list(reqs)
    qh = q.detach().cpu()
    pt, sl = page_table.cpu(), seq_lens.cpu()
    n = min(host_threads(), len(reqs))
    groups = [reqs[i::n] for i in range(n)]

    def run(g):
        return orc.decode(qh[g], k_host, v_host, pt[g], sl[g], sm_scale)

    with ThreadPoolExecutor(n) as ex:
        res = list(ex.map(run, groups))
    Hq, d = qh.shape[1], qh.shape[2]
    out = np.zeros((len(reqs), Hq, d), dtype=np.float64)
    lse = np.zeros((len(reqs), Hq), dtype=np.float64)
    pos = {r: i for i, r in enumerate(reqs)}
    for g, (o, l) in zip(groups, res):
        idx = [pos[r] for r in g]
        out[idx] = o
        lse[idx] = l
    return out, lse


def parallel_oracle_extend(k_host, v_host, q, page_table, cached_lens, extend_lens, q_offsets,
                           sm_scale, chunk: int = 64):
    """Oracle extend of every new token of a batch, on one thread per host
    core.  New tokens t0 .. t1-1 of a request with C cached tokens are the
    extend of t1 - t0 tokens over C + t0 cached ones (each sees positions
    0 .. C + t by definition), so each request is cut into pieces of `chunk`
    tokens and the pieces are spread over the threads; every piece is one
    call of the single-threaded C oracle.  Returns out [T, H_q, d] float64."""
    orc = oracle.get()
    qh = q.detach().cpu()
    pt = page_table.cpu()
    cl, el, qo = cached_lens.tolist(), extend_lens.tolist(), q_offsets.tolist()
    pieces = []
    for r, (C, E) in enumerate(zip(cl, el)):
        for t0 in range(0, E, chunk):
            pieces.append((r, C, t0, min(E, t0 + chunk)))
    pieces.sort(key=lambda p: -(p[1] + p[3]) * (p[3] - p[2]))  # longest first

    def run(p):
        r, C, t0, t1 = p
        a = qo[r] + t0
        return a, orc.extend(qh[a:a + t1 - t0], k_host, v_host, pt[r:r + 1],
                             torch.tensor([C + t0], dtype=torch.int32),
                             torch.tensor([t1 - t0], dtype=torch.int32), sm_scale)

    T, Hq, d = qh.shape
    out = np.zeros((T, Hq, d), dtype=np.float64)
    with ThreadPoolExecutor(host_threads()) as ex:
        for a, o in ex.map(run, pieces):
            out[a:a + o.shape[0]] = o
    return out
