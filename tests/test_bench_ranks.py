"""The multi-GPU timing logic of bench.py on CPU: two gloo ranks, each with its
own elapsed time; every rank must see the slowest one, and the job's rate is
all ranks' units over that time (weak scaling, no data-path collective)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [7.5, 9.25][rank]
        slowest = bench.max_over_ranks(mine, dist)
        rate = bench.job_throughput(4096 * 4096, 10, world, slowest * 1e-3)
        out.put((rank, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [9.25, 9.25]
    want = 2 * 4096 * 4096 * 10 / 9.25e-3
    assert res[0][2] == pytest.approx(want) and res[1][2] == pytest.approx(want)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(100, 2, 1, 4.0) == 50.0
