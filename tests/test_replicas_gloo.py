"""The N > 1 path of bench.py (independent replicas, no data-path collective):
world-size-2 gloo process group on CPU.  The job's step time is the slowest
rank's and its throughput counts every replica's work."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = [0.30, 0.45][rank]
    got = bench.slowest_rank_ms(ms, "cpu")
    dist.barrier()
    q.put((rank, got, bench.job_throughput(1e9, world, got)))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [0.45, 0.45]
    assert all(abs(o[2] - 2 * 1e9 / 0.45e-3 / 1e9) < 1e-6 for o in out)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.slowest_rank_ms(0.25, "cpu") == 0.25
    assert bench.job_throughput(2e9, 1, 1.0) == 2000.0
