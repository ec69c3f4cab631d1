"""minisgl_check_indices on the GPU: it counts exactly the out-of-range index
values that a decode or extend call over the same tensors would read (and
no entry past a request's length), against a plain count on the host."""
import pytest
import torch

import paged_kv_cache_row_gb300 as mk
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_row_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def host_counts(pt, lens, out_loc, num_rows):
    W = pt.shape[1]
    bad_pt = bad_loc = bad_len = 0
    for r in range(pt.shape[0]):
        n = int(lens[r])
        bad_len += int(n < 0 or n > W)
        for j in range(min(max(n, 0), W)):
            v = int(pt[r, j])
            bad_pt += int(v < 0 or v >= num_rows)
    for v in out_loc.tolist():
        bad_loc += int(v < 0 or v >= num_rows)
    return [bad_pt, bad_loc, bad_len]


def test_clean_decode_workload_counts_nothing():
    case = workloads.decode_llama3_8b(num_layers=1)  # padding requests and NaN-row padding columns
    counts = mk.minisgl_check_indices(case.page_table.to(DEV), case.seq_lens.to(DEV), case.num_rows,
                                      out_loc=case.out_loc.to(DEV))
    assert counts.cpu().tolist() == [0, 0, 0]


def test_planted_bad_entries_are_counted_exactly():
    case = workloads.make_decode_case("bad-idx", num_layers=1, num_q_heads=8, num_kv_heads=2,
                                      head_dim=64, page_size=1, batch=9, ctx_lo=5, ctx_hi=300,
                                      num_dummy=2, dummy_seq_len=3, seed=21)
    pt, lens, loc = case.page_table.clone(), case.seq_lens.clone(), case.out_loc.clone()
    R = case.num_rows
    g = torch.Generator().manual_seed(4)
    for i in range(40):  # inside the read range: counted (a cell hit twice counts once)
        r = int(torch.randint(0, case.batch, (1,), generator=g))
        j = int(torch.randint(0, int(lens[r]), (1,), generator=g))
        pt[r, j] = R + int(torch.randint(0, 5, (1,), generator=g)) if i % 2 else -1 - i
    pt[0, int(lens[0]):] = -7  # past the length: never read, not counted
    loc[3], loc[5] = R, -2
    lens[6] = pt.shape[1] + 1  # longer than the page-table width
    counts = mk.minisgl_check_indices(pt.to(DEV), lens.to(DEV), R, out_loc=loc.to(DEV))
    assert counts.cpu().tolist() == host_counts(pt, lens, loc, R)
    assert counts.cpu().tolist()[2] == 1
    # a second call on the same counts tensor starts from zero
    again = mk.minisgl_check_indices(pt.to(DEV), lens.to(DEV), R, out_loc=loc.to(DEV), counts=counts)
    assert again.cpu().tolist() == host_counts(pt, lens, loc, R)


def test_extend_lengths_and_empty_inputs():
    case = workloads.make_extend_case("idx-ext", num_q_heads=8, num_kv_heads=2, head_dim=128,
                                      num_reqs=4, prefix_len=50, ext_lo=10, ext_hi=90, budget=128,
                                      seed=5)
    for b in case.batches:
        lens = (b.cached_lens + b.extend_lens).to(torch.int32)
        counts = mk.minisgl_check_indices(b.page_table.to(DEV), lens.to(DEV), case.num_rows,
                                          out_loc=b.out_loc.to(DEV))
        assert counts.cpu().tolist() == [0, 0, 0]
    empty = torch.empty((0, 32), dtype=torch.int32, device=DEV)
    counts = mk.minisgl_check_indices(empty, torch.empty(0, dtype=torch.int32, device=DEV), 10)
    assert counts.cpu().tolist() == [0, 0, 0]


def host_shared_prefix_counts(pt, lens, P):
    diff = sum(int(pt[r, j] != pt[0, j]) for r in range(1, pt.shape[0]) for j in range(P))
    short = sum(int(int(n) < P) for n in lens.tolist())
    return [diff, short]


def test_shared_prefix_check():
    """minisgl_check_shared_prefix counts the prefix entries that differ from
    the first request's and the requests shorter than the prefix: none on a
    radix-shared batch, exactly the planted ones after corrupting it, and it
    agrees with a host count when the declared prefix is longer than the
    shared one."""
    case = workloads.make_shared_prefix_decode_case("check-shared", num_q_heads=8, num_kv_heads=2,
                                                    head_dim=128, batch=9, prefix_len=300,
                                                    suffix_lo=0, suffix_hi=50, seed=5)
    pt, sl = case.page_table.clone(), case.seq_lens.clone()
    got = mk.minisgl_check_shared_prefix(pt.to(DEV), sl.to(DEV), 300)
    assert got.cpu().tolist() == [0, 0]
    pt[3, 17] += 1
    pt[8, 299] = case.num_rows - 1
    sl[2] = 299
    got = mk.minisgl_check_shared_prefix(pt.to(DEV), sl.to(DEV), 300)
    assert got.cpu().tolist() == [2, 1] == host_shared_prefix_counts(pt, sl, 300)
    P = int(pt.shape[1])  # declared longer than what is shared
    got = mk.minisgl_check_shared_prefix(pt.to(DEV), sl.to(DEV), P)
    assert got.cpu().tolist() == host_shared_prefix_counts(pt, sl, P)
