"""Helpers shared by the GPU parity tests (marshalling and comparisons only).

Oracle inputs are always the generator's values copied from the device BEFORE
any library kernel runs; new rows reach the oracle's copy of the pool through
the oracle's own store_kv, never through the CUDA path's output.
"""
from __future__ import annotations

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
