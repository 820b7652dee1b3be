"""The benchmark's multi-rank arithmetic on CPU (gloo, world size 2): the job's
time is the slowest rank's, and throughput counts the units of every rank.
With N GPUs each rank decodes its own batch (weak scaling, no data collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    bench.dist_init(w, "gloo")
    elapsed = [0.5, 0.8][r]                      # seconds measured on this rank
    bench.barrier(w)
    slowest = bench.max_over_ranks(elapsed, w)
    value = bench.aggregate_throughput(8 * 10, w, slowest)
    q.put((r, w, local, slowest, value))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_ranks_max_time_and_whole_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, (rank, world, local, slowest, value) in enumerate(res):
        assert (rank, world, local) == (r, 2, r)
        assert slowest == pytest.approx(0.8)
        assert value == pytest.approx(8 * 10 * 2 / 0.8)


def test_single_rank_defaults():
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.aggregate_throughput(100, 1, 0.5) == 200
