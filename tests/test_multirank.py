"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2):
token data parallelism with no data-path exchange; the job's time is the
slowest rank's and the throughput counts every rank's tokens."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_info() == (world, rank, rank)
        local_seconds = [0.010, 0.025][rank]
        slowest = bench.max_over_ranks(local_seconds, world, "cpu")
        out[rank] = (slowest, bench.job_throughput(world, 512, 100, slowest))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_over_ranks_and_throughput():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        slowest, value = out[r]
        assert slowest == pytest.approx(0.025)
        assert value == pytest.approx(2 * 512 * 100 / 0.025)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.job_throughput(1, 512, 10, 2.0) == 2560.0
