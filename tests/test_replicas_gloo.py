"""The N > 1 bench path on CPU: world-size-2 gloo process groups check the
max-over-ranks timing and the whole-job rate that bench.py reports (replicas
only: each rank decodes its own stream, no data-path collective)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ws, r, local = bench.dist_env()
        seconds = 1.0 + rank  # rank 1 is the slow one
        tmax = bench.max_over_ranks(seconds)
        rate = bench.whole_job_rate(256, ws, tmax)
        q.put((rank, ws, r, local, tmax, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ws, r, local, tmax, rate in got:
        assert ws == 2 and r == rank and local == rank
        assert tmax == 2.0  # the slowest rank's time on every rank
        assert rate == 2 * 256 / 2.0


def test_single_process_helpers():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(100, 1, 0.5) == 200.0
    assert bench.LAUNCHES_PER_TOKEN[3] == 1
