"""The benchmark's multi-rank path on CPU: two gloo ranks on 127.0.0.1.

Each rank runs its own batch with no collective on the data path; the only
cross-rank steps are the barriers around the timed region and the maximum of
the ranks' times, from which the whole-job rate is computed.  Here each rank
reports a different time and must end up with the slowest one, and the job
rate must count both ranks' units.  No GPU is used.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    w, r, local = bench.dist_setup(world, backend="gloo")
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    my_ms = 2.0 + 3.0 * rank          # rank 0: 2 ms, rank 1: 5 ms
    ms = bench.max_over_ranks(my_ms, w)
    rate = bench.job_rate(1000.0, w, ms)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    out.put((rank, ms, rate))


@pytest.mark.timeout(300)
def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(240)
        assert p.exitcode == 0, f"rank process exited with {p.exitcode}"
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, rate in res:
        assert ms == 5.0, (rank, ms)                 # both ranks see the slowest rank
        assert rate == pytest.approx(2 * 1000.0 / 5e-3)  # both ranks' units over that time


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_rate(10.0, 1, 2.0) == pytest.approx(5000.0)
