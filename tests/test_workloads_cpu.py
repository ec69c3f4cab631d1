"""Structure of the synthetic inputs the benchmark's newer objects use,
checked on the CPU: the mixed chunk + decode batch and the store_kv rotation."""
import torch

import workloads


def test_mixed_batch_structure():
    mc = workloads.mixed_chunk_decode()
    b = mc.batches[0]
    base = workloads.extend_radix_shared().batches[0]
    nd = mc.num_decode
    nb = len(b.req_ids) - nd
    assert nb == len(base.req_ids) and nd == 64
    # the chunk part is the radix-shared workload's first batch, unchanged
    assert torch.equal(b.cached_lens[:nb], base.cached_lens)
    assert torch.equal(b.extend_lens[:nb], base.extend_lens)
    Tc = int(b.q_offsets[nb])
    assert Tc == base.total_tokens and torch.equal(b.out_loc[:Tc], base.out_loc)
    # decode requests: one new token over U[512, 4096] cached ones, stored in the
    # row their page table names for that position
    assert bool((b.extend_lens[nb:] == 1).all())
    assert int(b.cached_lens[nb:].min()) >= 512 and int(b.cached_lens[nb:].max()) <= 4096
    for k in range(nd):
        C = int(b.cached_lens[nb + k])
        assert int(b.out_loc[Tc + k]) == int(b.page_table[nb + k, C])
    # decode requests' rows are their own and inside the live pool
    rows = torch.cat([b.page_table[nb + k, :int(b.cached_lens[nb + k]) + 1] for k in range(nd)])
    assert rows.unique().numel() == rows.numel()
    assert int(rows.max()) < mc.num_rows - 2 and int(rows.min()) >= workloads.extend_radix_shared().num_rows - 2
    assert b.page_table.shape[1] % 32 == 0


def test_store_rotation_rows_are_disjoint():
    rot = workloads.store_rotation(batches=4, tokens=512)
    allrows = torch.cat(rot.out_locs)
    assert allrows.numel() == 4 * 512 and allrows.unique().numel() == allrows.numel()
    assert int(allrows.min()) >= 0 and int(allrows.max()) < rot.num_rows - 2
