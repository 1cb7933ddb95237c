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


def test_phase_rooflines_scale_with_time():
    """Achieved rates are work / time: halving a phase's time doubles its
    rate; fractions are achieved / peak with the stated peaks; the prepare
    step's GEMM share is quoted against the measured 3xTF32 rate."""
    import bench
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 1800.0, "source": "test"}
    box = {"tf32_tflops": 900.0, "tf32x3_tflops": 300.0, "fp32_tflops": 70.0}
    ph = {"prepare": 2.0, "quantize": 1.0, "pack": 0.1}
    a = bench.phase_rooflines(ph, 4096, 4096, 4, 128, peaks, box=box, prep_gemm_ms=0.5)
    b = bench.phase_rooflines({k: v / 2 for k, v in ph.items()}, 4096, 4096, 4, 128, peaks, box=box,
                              prep_gemm_ms=0.25)
    for k in ("quantize", "pack"):
        assert abs(b[k]["achieved"] / a[k]["achieved"] - 2.0) < 1e-3
        assert abs(a[k]["frac"] - a[k]["achieved"] / a[k]["peak"]) < 1e-3
    g = a["prepare"]["gemm"]
    assert abs(b["prepare"]["gemm"]["achieved"] / g["achieved"] - 2.0) < 2e-3
    assert g["peak"] == 300.0 and abs(g["frac"] - g["achieved"] / 300.0) < 1e-3
    assert abs(a["prepare"]["panel_ms"] - 1.5) < 1e-9
    # pack: 1.5 B/weight in 0.1 ms; quantize against the measured 3xTF32 rate
    assert abs(a["pack"]["achieved"] - 4096 * 4096 * 1.5 / 1e-4 / 1e9) < 0.1
    assert a["quantize"]["peak"] == 300.0


def test_prepare_gemm_flops_is_the_lower_triangle_count():
    """Replayed update GEMM flops: brute-force count of the lower-triangle
    elements each step updates, 2 * K flops each; about 2 d^3 / 3 in all."""
    import bench
    d, nb = 512, 128
    want = 0
    for k in range(0, d - nb, nb):
        for i in range(k + nb, d):
            want += 2 * nb * (i + 1)
    assert bench.prepare_gemm_flops(d, nb) == want
    assert abs(bench.prepare_gemm_flops(4096) / (2 * 4096 ** 3 / 3) - 1) < 0.05
