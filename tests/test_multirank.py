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


def test_rank_seeds_are_disjoint():
    """Every rank draws its own batch and weights: the three seeds of each
    (layer, rank) never coincide with another's."""
    import bench
    seen = {}
    for rank in range(8):
        for layer in range(64):
            s = bench.layer_seed(layer, rank)
            for off in range(3):
                assert (s + off) not in seen, (layer, rank, seen.get(s + off))
                seen[s + off] = (layer, rank)


def test_bench_gpus_flag_launches_ranks():
    """`bench.py --gpus 2` outside a launcher runs itself as two ranks under
    torch.distributed.run (gloo here, no GPU: the reference arm, which rank 0
    alone runs and prints); the line reports n_gpus = 2 and both ranks exit 0."""
    import json
    import subprocess
    import sys
    from pathlib import Path
    root = Path(__file__).resolve().parent.parent
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, str(root / "bench.py"), "--impl", "reference", "--gpus",
                        "2", "--workload", "small", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, env=env, cwd=str(root))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    assert out["n_gpus"] == 2 and out["impl"] == "reference" and out["steps"] == 1
