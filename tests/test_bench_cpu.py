"""The benchmark's roofline arithmetic, checked on the CPU.

bench.py reports achieved GB/s and TFLOP/s as algorithmic work per call over
the measured time.  These tests recount that work by brute force on small
seeded cases (every page-table position, every causal query/key pair) and
compare it with the closed forms bench.py uses, so a dropped term or an
off-by-one in a formula shows up here rather than as a wrong roofline
fraction.  They also check the rule that a committed ncu traffic figure is
only reported while the kernel source it was taken on is unchanged.
"""
import hashlib
import os

import pytest

import bench
import workloads


def _decode_case(num_dummy=0, page_size=1, seed=5):
    return workloads.make_decode_case("bytes", num_layers=1, num_q_heads=8, num_kv_heads=2,
                                      head_dim=64, page_size=page_size, batch=7, ctx_lo=3,
                                      ctx_hi=90, num_dummy=num_dummy, dummy_seq_len=5, seed=seed)


def _brute_decode_bytes(case):
    """Every K/V row a decode call must read (a row several requests read
    counts once), every page-table entry read, queries, outputs, seq_lens."""
    Hkv, d, Hq = case.num_kv_heads, case.head_dim, case.num_q_heads
    rows, entries = set(), 0
    for r in range(case.batch):
        n = int(case.seq_lens[r])
        for j in range(n):
            rows.add(int(case.page_table[r, j]))
            entries += 1
    return (len(rows) * 2 * Hkv * d * 2 + entries * 4 + case.batch * Hq * d * 2 * 2
            + case.batch * 4)


@pytest.mark.parametrize("num_dummy,page_size", [(0, 1), (3, 1), (0, 64)])
def test_decode_bytes_match_enumeration(num_dummy, page_size):
    case = _decode_case(num_dummy=num_dummy, page_size=page_size)
    assert bench.decode_layer_bytes(case) == _brute_decode_bytes(case)


def test_store_bytes_match_enumeration():
    case = _decode_case()
    Hkv, d = case.num_kv_heads, case.head_dim
    brute = 0
    for _ in range(case.batch):  # read k and v, write both into the pool, read out_loc
        brute += 2 * (Hkv * d * 2) + 2 * (Hkv * d * 2) + 4
    assert bench.store_layer_bytes(case) == brute


def test_cascade_bytes_match_enumeration():
    case = workloads.make_shared_prefix_decode_case("cascade-bytes", num_q_heads=8, num_kv_heads=2,
                                                    head_dim=64, batch=5, prefix_len=40,
                                                    suffix_lo=1, suffix_hi=30, seed=3)
    Hkv, d, Hq = case.num_kv_heads, case.head_dim, case.num_q_heads
    rows = set()
    for r in range(case.batch):
        rows.update(int(x) for x in case.page_table[r, :int(case.seq_lens[r])])
    # the shared rows and their entries once, each private row and entry once
    brute = len(rows) * (2 * Hkv * d * 2 + 4) + case.batch * Hq * d * 2 * 2 + case.batch * 4
    assert bench.cascade_layer_bytes(case) == brute


def test_extend_flops_match_pair_count():
    case = workloads.make_extend_case("flops", num_q_heads=4, num_kv_heads=2, head_dim=64,
                                      num_reqs=5, prefix_len=37, ext_lo=3, ext_hi=70, budget=96,
                                      seed=11)
    assert len(case.batches) > 1  # a request is cut across batches
    pairs = 0
    for b in case.batches:
        for C, E in zip(b.cached_lens.tolist(), b.extend_lens.tolist()):
            for t in range(E):          # new token t sits at position C + t ...
                for _j in range(C + t + 1):  # ... and sees positions 0 .. C + t
                    pairs += 1
    # per (query head, visible key): q.k and p.v, d multiply-adds each
    assert bench.extend_flops(case) == pytest.approx(pairs * case.num_q_heads * 4 * case.head_dim,
                                                     rel=0, abs=0)


def test_job_rate_counts_every_rank():
    assert bench.job_rate(1000.0, 1, 2.0) == pytest.approx(500000.0)
    assert bench.job_rate(1000.0, 4, 2.0) == pytest.approx(2000000.0)
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_profile_traffic_only_for_the_profiled_source(tmp_path, monkeypatch):
    src_dir = tmp_path / "paged_kv_cache_row_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = src_dir / "k.cu"
    src.write_bytes(b"__global__ void k() {}\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles" / "k.md").write_text(
        f"kernel_source_sha256_16: {digest}\ntraffic_bytes_per_launch: 12345\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic("k.cu", "k.md") == 12345.0
    src.write_bytes(b"__global__ void k() { /* changed */ }\n")
    assert bench.profile_traffic("k.cu", "k.md") is None
    assert bench.profile_traffic("k.cu", "missing.md") is None


def test_committed_profiles_name_their_sources():
    """Every committed profile that gives a per-launch traffic figure also
    names the kernel source version it was taken on."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    prof = os.path.join(root, "profiles")
    for name in os.listdir(prof):
        text = open(os.path.join(prof, name)).read()
        if "traffic_bytes_per_launch" in text:
            assert "kernel_source_sha256_16" in text, name


@pytest.mark.parametrize("L", [1, 2, 3, 5, 28, 32, 33, 64])
def test_e2e_input_waits_cover_every_layer(L):
    """Before each layer runs, some earlier (or its own) wait covers its inputs,
    and no wait points past the last layer."""
    sched = bench.input_wait_schedule(L)
    assert 0 in sched and sched[0] >= 0
    covered = -1
    for layer in range(L):
        if layer in sched:
            assert layer <= sched[layer] <= L - 1
            covered = max(covered, sched[layer])
        assert covered >= layer, (L, layer)
    assert len(sched) <= L.bit_length() + 1
