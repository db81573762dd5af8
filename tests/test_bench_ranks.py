"""The bench's multi-rank host logic on CPU, with two gloo ranks: the step time
is the slowest rank's on every rank, and the whole-job rate counts every
rank's replica against that time (weak scaling).  Sequences are independent,
so the GPU path has no exchange step; these are the only cross-rank values."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
torch = pytest.importorskip("torch")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench._max_over_ranks(times[rank], "cpu")
        out.put((rank, ms, bench._job_rate(1000.0, ms, world), bench._dist()))
    finally:
        dist.destroy_process_group()


def test_step_time_is_the_slowest_rank_and_rate_counts_every_replica():
    ctx = torch.multiprocessing.get_context("spawn")
    out = ctx.Queue()
    times = [0.25, 0.40]
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate, dist_env in got:
        assert ms == 0.40                                   # the slowest rank's time, on both ranks
        assert rate == pytest.approx(2 * 1000.0 / 0.40e-3)  # both replicas' units over that time
        assert dist_env == (2, rank, rank)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._max_over_ranks(0.3, "cpu") == 0.3
    assert bench._job_rate(500.0, 0.5, 1) == pytest.approx(1e6)
