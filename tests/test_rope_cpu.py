"""Host-side pieces of the RoPE step: the cos/sin table the engine builds and
the token positions the workloads hand to it (no GPU)."""
import math

import numpy as np
import torch

import workloads


def test_cos_sin_table_closed_form():
    # d = 4, base 10000: frequencies 1 and 10000^(-1/2) = 0.01
    t = workloads.rope_cos_sin_cache(4, 3)
    assert t.dtype == torch.float32 and t.shape == (3, 4)
    want = np.array([[1.0, 1.0, 0.0, 0.0],
                     [math.cos(1.0), math.cos(0.01), math.sin(1.0), math.sin(0.01)],
                     [math.cos(2.0), math.cos(0.02), math.sin(2.0), math.sin(0.02)]])
    assert np.abs(t.numpy() - want).max() <= 2e-7


def test_cos_sin_table_layout_d128():
    t = workloads.rope_cos_sin_cache(128, 50, base=1e6)
    f = 1e6 ** (-np.arange(0, 128, 2) / 128.0)
    ang = np.outer(np.arange(50), f)
    ref = np.concatenate([np.cos(ang), np.sin(ang)], 1)
    # float32 angles: |error| <= position * ulp(freq) plus the rounding of cos/sin
    assert np.abs(t.numpy() - ref).max() <= 5e-6


def test_extend_positions_follow_cached_lens():
    case = workloads.extend_radix_shared()
    for b in case.batches:
        pos = workloads.extend_positions(b)
        assert pos.dtype == torch.int32 and pos.numel() == b.total_tokens
        for r, (c, e) in enumerate(zip(b.cached_lens.tolist(), b.extend_lens.tolist())):
            o = int(b.q_offsets[r])
            assert torch.equal(pos[o:o + e], torch.arange(c, c + e, dtype=torch.int32))


def test_decode_positions_and_padding():
    case = workloads.decode_llama3_8b(num_layers=1)
    pos = workloads.decode_positions(case)
    n = case.num_real
    assert torch.equal(pos[:n], (case.seq_lens[:n] - 1).to(torch.int32))
    assert bool((pos[n:] == 0).all())
