"""Benchmark: GPTQ layer solve on one 7B attention projection per GPU.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload (per GPU): W bf16 4096 x 4096 ~ N(0, 0.02^2); calibration X fp16
4096 x 262144 (128 sequences x 2048 tokens) ~ N(0, 1) with 1% of channels
scaled by U[10, 50]; 4-bit asymmetric, group 128, damp 0.01, blocksize 128,
desc_act off.  A step is one pass of the whole solver on that layer:
S = 0; S += X X^T; prepare H^-1 factor; quantize; pack.  The inputs are
resident in HBM when the timed region starts; X (2.15 GB) is larger than
L2, so no extra flush is needed.

Prints one JSON line (rank 0).  Metric: weights quantized per second
(Mweights/s), whole job.  With torchrun (N > 1) every rank solves its own
layer (weak scaling, no collective on the data path); the time is the max
over ranks.

The line also carries "dequant": gptq_dequantize of the solved layer's
packed output to fp16, timed per launch with an L2 flush (the consumer of the
packed format).  --dequant-only ROWSxCOLS times that kernel alone on a random
packed 4-bit g128 layer of the given shape (bf16 output).

--impl reference times the CPU oracle (the same algorithm in NumPy fp64) on
a bounded sample of the same workload and extrapolates to the full layer.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

D = 4096
N_TOK = 262144
METRIC = "GPTQ layer-solve Mweights/s (4096x4096, 4-bit g128)"
WORKLOAD = ("7B attention projection: W bf16 4096x4096 N(0,0.02^2); X fp16 4096x262144 "
            "N(0,1), 1% channels x U[10,50]; 4-bit asym g128, damp 0.01, blocksize 128, "
            "desc_act off")


# DRAM bytes (read + write) of one hessian_syrk_kernel launch at the full
# workload, from a one-pass ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum).  It describes the kernel source it was measured on
# (sha256 prefixes below); once that source changes the figure no longer
# applies and the bench reports null.
SYRK_TRAFFIC = {"bytes": 5.948e9, "n_tok": 262144,
                "sha256": {"hessian_syrk.cu": "8ceb7328e0e05e8a", "common.cuh": "e1bfb68f46b7876c"}}


def syrk_traffic() -> float | None:
    import hashlib
    if N_TOK != SYRK_TRAFFIC["n_tok"]:
        return None
    csrc = os.path.join(ROOT, "post_weight_quantization_31_b300", "csrc")
    for name, want in SYRK_TRAFFIC["sha256"].items():
        with open(os.path.join(csrc, name), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != want:
                return None
    return SYRK_TRAFFIC["bytes"]


def set_tokens(n: int) -> None:
    """Shrinks the calibration set (profiling cases only)."""
    global N_TOK, WORKLOAD
    WORKLOAD = WORKLOAD.replace(f"4096x{N_TOK}", f"4096x{n}") + " (profiling case)"
    N_TOK = n


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples during the timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def mark(self, which: str) -> None:
        """Wall-clock bounds of the timed region (samples outside are dropped)."""
        setattr(self, which, time.time())

    def summary(self) -> dict:
        import datetime
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append(dict(ts=ts, sm=float(parts[2]), smax=float(parts[3]), active=parts[5],
                                 hw=parts[6], hwt=parts[7], swt=parts[8], pcap=parts[9]))
            except ValueError:
                continue
        t0, t1 = getattr(self, "start", None), getattr(self, "end", None)
        if rows and t0 is not None and t1 is not None:
            inside = [r for r in rows if t0 - 0.05 <= r["ts"] <= t1 + 0.05]
            rows = inside or sorted(rows, key=lambda r: abs(r["ts"] - 0.5 * (t0 + t1)))[:1]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows)}


# ---------------------------------------------------------------- ranks
def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The largest x over all ranks (the job ends when its slowest rank ends)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, steps: int, world: int, seconds: float) -> float:
    """Whole-job rate: every rank processes its own units (weak scaling)."""
    return world * units_per_rank * steps / seconds


# ---------------------------------------------------------------- peaks
def measure_box_peaks(dev) -> dict:
    """Dense GEMM rates of the types the solve uses, measured here with
    cuBLAS (torch.matmul, 8192^3, best of 5 after warm-up, CUDA events):
    TF32 (fp32 inputs with TF32 allowed) and FP32 (TF32 off).  3xTF32 does
    three TF32 products per output term, so its peak is TF32 / 3."""
    import torch
    n = 8192
    a = torch.randn((n, n), device=dev)
    b = torch.randn((n, n), device=dev)
    out = {}
    old = torch.backends.cuda.matmul.allow_tf32
    try:
        for name, tf32 in (("tf32_tflops", True), ("fp32_tflops", False)):
            torch.backends.cuda.matmul.allow_tf32 = tf32
            for _ in range(2):
                torch.matmul(a, b)
            best = float("inf")
            for _ in range(5):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                torch.matmul(a, b)
                e1.record()
                torch.cuda.synchronize(dev)
                best = min(best, e0.elapsed_time(e1))
            out[name] = round(2.0 * n ** 3 / (best * 1e-3) / 1e12, 1)
    finally:
        torch.backends.cuda.matmul.allow_tf32 = old
    out["tf32x3_tflops"] = round(out["tf32_tflops"] / 3.0, 1)
    out["how"] = "cuBLAS via torch.matmul 8192^3, best of 5 (CUDA events), this run"
    return out


def prepare_gemm_ms(d: int, dev, reps: int = 3) -> float:
    """Time of the prepare step's update GEMMs alone: the same 3xTF32
    launches (M = d - k - 128 rows, N = d lower, K = 128, for every step k)
    replayed through the library's GEMM on synthetic operands, CUDA events
    around all of them, best of `reps`.  The prepare time minus this is the
    panel (factorization) share."""
    import ctypes

    import torch
    from post_weight_quantization_31_b300 import _lib
    lib = _lib.load()
    f = lib.gptq_internal_tgemm
    f.restype = ctypes.c_int
    vp, i64, i32, fl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    f.argtypes = [vp, vp, i64, vp, vp, i64, i32, i32, i32, fl, fl, vp, i64, i32, i32, i32, vp]
    nb = 128
    Bh = torch.randn((d, nb), device=dev) * 1e-3
    Bl = torch.zeros_like(Bh)
    Z = torch.zeros((d, d), device=dev)
    st = torch.cuda.current_stream(dev).cuda_stream
    best = float("inf")
    for _ in range(reps + 1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for k in range(0, d - nb, nb):
            r = k + nb
            rc = f(Bh[r:].data_ptr(), Bl[r:].data_ptr(), nb, Bh.data_ptr(), Bl.data_ptr(), nb, d - r, d, nb,
                   -1.0, 1.0, Z[r:].data_ptr(), d, 1, r, 0, st)
            if rc != 0:
                raise RuntimeError(f"gptq_internal_tgemm failed: {rc}")
        e1.record()
        torch.cuda.synchronize(dev)
        best = min(best, e0.elapsed_time(e1))
    return best


def prepare_gemm_flops(d: int, nb: int = 128) -> float:
    """Flops of those update GEMMs: for step k, rows r >= k + nb, columns
    c <= r (lower), K = nb, 2 flops per multiply-add."""
    tot = 0.0
    for k in range(0, d - nb, nb):
        r = k + nb
        rows = d - r
        # sum over rows i in [r, d) of (i + 1) columns
        tot += 2.0 * nb * (rows * (r + d + 1) / 2.0)
    return tot


def phase_rooflines(ph_ms: dict, d_row: int, d_col: int, bits: int, group_size: int,
                    peaks: dict, box: dict | None = None, prep_gemm_ms: float | None = None,
                    block: int = 128) -> dict:
    """Roofline fraction of each solve phase from its CUDA-event time and its
    algorithmic work, each against the measured peak of the unit it runs on:
      prepare   its update GEMMs (3xTF32 on the tensor cores) against the
                measured 3xTF32 rate, over their own replayed time; the rest
                of the phase (the panel factorizations, a latency chain) is
                reported as time only;
      quantize  the trailing updates' d_row·d_col·(d_col − B) flop against
                the 3xTF32 rate, over the phase time; the column loop inside
                the same phase moves read W (2 B) + codes (bits/8 B) +
                scale/zero (5 B per group element) per weight, reported
                against HBM;
      pack      1 + bits/8 B per weight against HBM."""
    hbm = float(peaks.get("hbm_gbs", 6400.0))
    if box:
        tf32_3x, src = float(box["tf32x3_tflops"]), "measured cuBLAS TF32 / 3"
    else:
        tf32_3x, src = float(peaks.get("bf16_tflops", 1800.0)) / 2.0 / 3.0, "nominal (bf16 / 2 / 3)"
    W = float(d_row) * d_col
    G = 1 if group_size == -1 else d_col // group_size
    out = {}
    t = ph_ms.get("prepare")
    if t:
        entry = {"ms": round(t, 4)}
        if prep_gemm_ms:
            fl = prepare_gemm_flops(d_col)
            a = fl / (prep_gemm_ms * 1e-3) / 1e12
            entry.update({"gemm": {"bound": "tensor", "ms": round(prep_gemm_ms, 4), "flop": fl,
                                   "achieved": round(a, 1), "peak": tf32_3x, "unit": "TFLOP/s",
                                   "frac": round(a / tf32_3x, 4)},
                          "panel_ms": round(max(t - prep_gemm_ms, 0.0), 4),
                          "panel_note": "diagonal-block factorizations: a latency chain, time only"})
        out["prepare"] = entry
    t = ph_ms.get("quantize")
    if t:
        a = W * max(d_col - block, 0) / (t * 1e-3) / 1e12
        col_bytes = W * (2.0 + bits / 8.0) + 5.0 * G * d_row
        b = col_bytes / (t * 1e-3) / 1e9
        out["quantize"] = {"bound": "tensor", "achieved": round(a, 2), "peak": tf32_3x,
                           "unit": "TFLOP/s", "frac": round(a / tf32_3x, 4),
                           "column_loop_bytes": int(col_bytes), "column_loop_gbs": round(b, 1),
                           "column_loop_frac_of_hbm": round(b / hbm, 4)}
    t = ph_ms.get("pack")
    if t:
        b = W * (1.0 + bits / 8.0) / (t * 1e-3) / 1e9
        out["pack"] = {"bound": "hbm", "achieved": round(b, 1), "peak": hbm, "unit": "GB/s",
                       "frac": round(b / hbm, 4)}
    out["peak_note"] = (f"HBM: {peaks.get('source', 'fallback')} copy bandwidth; 3xTF32: {src}")
    return out


def make_inputs():
    from post_weight_quantization_31_b300 import workloads as wl
    return wl.attn_proj_7b(seed=1002, n_tok=N_TOK, d=D)


# ---------------------------------------------------------------- our arm
def run_ours(args, rank: int, world: int, local_rank: int) -> dict | None:
    import torch
    from post_weight_quantization_31_b300 import api, build_lib

    build_lib.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    inp = make_inputs()
    cfg = inp.cfg
    X = torch.from_numpy(inp.X).to(dev)
    W = torch.from_numpy(inp.W).to(torch.bfloat16).to(dev)
    solver = api.LayerSolver(D, D, cfg, device=dev, exact_diag=False)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        solver.reset()
        if ev is not None:
            ev[0].record(stream)
        solver.accumulate(X)
        if ev is not None:
            ev[1].record(stream)
        solver.prepare()
        if ev is not None:
            ev[2].record(stream)
        solver.quantize(W)
        if ev is not None:
            ev[3].record(stream)
        solver.pack()
        if ev is not None:
            ev[4].record(stream)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    # The sampler starts before the warm-up so that it is running when the
    # timed region begins; only samples inside that region are kept.
    with ClockSampler(local_rank) as clk:
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        n0 = api.launch_count()
        clk.mark("start")
        t_start.record(stream)
        for k in range(args.steps):
            step(evs[k])
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        clk.mark("end")
    solver.check()      # device-side status of the last prepare / quantize
    if dist is not None:
        dist.barrier()
    launches = api.launch_count() - n0
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), dist, dev)

    ph = {name: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs)
          for i, name in enumerate(("hessian", "prepare", "quantize", "pack"))}

    # end to end through the public host-buffer API
    e2e = None
    if args.e2e_steps > 0:
        chunk = 32768
        chunks = [torch.from_numpy(np.ascontiguousarray(inp.X[:, a:a + chunk])).pin_memory()
                  for a in range(0, N_TOK, chunk)]
        W_host = torch.from_numpy(inp.W).to(torch.bfloat16).pin_memory()
        api.quantize_layer_from_host(W_host, chunks, cfg, solver=solver)  # warm
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            res = api.quantize_layer_from_host(W_host, chunks, cfg, solver=solver)
        torch.cuda.synchronize(dev)
        e2e_s = max_over_ranks(time.perf_counter() - t0, dist, dev)
        h2d = sum(c.numel() * c.element_size() for c in chunks) + W_host.numel() * 2
        d2h = sum(v.numel() * v.element_size() for v in res.values())
        e2e = {"value": round(job_throughput(D * D, args.e2e_steps, world, e2e_s) / 1e6, 3),
               "unit": "Mweights/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": args.e2e_steps}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return None

    box = measure_box_peaks(dev)
    prep_gemm = prepare_gemm_ms(D, dev)
    peaks = measured_peaks()
    syrk_ms = ph["hessian"]
    flops = float(N_TOK) * D * (D + 1)       # symmetric half of X X^T
    achieved = flops / (syrk_ms * 1e-3) / 1e12
    # The kernel is timed inside a 7 ms step, not a seconds-long loop, and the
    # step's clock samples sit at the maximum SM clock: the burst peak is the
    # denominator; the sustained (power-capped) one is given beside it.
    peak = float(peaks.get("bf16_tflops", 1800.0))
    sus = float(peaks.get("bf16_tflops_sustained", 1400.0))
    clocks = clk.summary()
    roof = {"kernel": "hessian_syrk_kernel (tcgen05 kind::f16, fp16 x fp16 -> fp32)",
            "bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4),
            "frac_of_sustained": round(achieved / sus, 4),
            "peak_note": (f"{peaks['source']} bf16 dense burst {peak} TFLOP/s (fp16 rate = bf16 rate), "
                          f"SM clock in the timed region {clocks.get('sm_mhz')} MHz; sustained "
                          f"{sus} TFLOP/s was measured at {peaks.get('clocks_under_load', {}).get('sm_mhz_median')} MHz"),
            "traffic": args.syrk_traffic if args.syrk_traffic is not None else syrk_traffic(),
            "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)"}
    ms_step = elapsed_ms / args.steps
    line = {
        "metric": METRIC,
        "value": round(job_throughput(D * D, args.steps, world, elapsed_ms * 1e-3) / 1e6, 3),
        "unit": "Mweights/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp16 x fp16 -> fp32 (Hessian), fp32 (solve)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "d_row": D, "d_col": D, "n_tok": N_TOK,
                   "l2": "inputs larger than L2 (X is 2.15 GB)",
                   "parallelism": f"one independent layer per GPU x{world}"},
        "phases_ms": {k: round(v, 4) for k, v in ph.items()},
        "phases_roofline": phase_rooflines(ph, D, D, cfg.bits, cfg.group_size, peaks, box=box,
                                           prep_gemm_ms=prep_gemm),
        "box_peaks": box,
        "solve_only": {"value": round(D * D / ((ph["prepare"] + ph["quantize"] + ph["pack"]) * 1e-3) / 1e6, 3),
                       "unit": "Mweights/s",
                       "note": "prepare + quantize + pack with H given, from the same timed steps"},
        "gpu_launches": int(launches),
        "roofline": roof,
        "clocks": clocks,
        "e2e": e2e,
    }
    if args.dequant_reps > 0:
        line["dequant"] = measure_dequant(solver, cfg, stream, peaks, args.dequant_reps)
    if args.layer_set_layers > 0:
        del X, W, solver
        torch.cuda.empty_cache()
        line["layer_set"] = measure_layer_set(layer_set_inputs(dev), args.layer_set_layers, dev)
    if args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, quick=args.quick_cpu)
    if dist is not None:
        dist.destroy_process_group()
    return line


class _OneRank:
    """torch.distributed stand-in for a single process (collectives are no-ops)."""

    class ReduceOp:
        SUM = "sum"

    @staticmethod
    def all_reduce(t, op=None, group=None):
        return None

    @staticmethod
    def broadcast(t, src=0, group=None):
        return None


def run_sharded(args, rank: int, world: int, local_rank: int) -> dict | None:
    """--shard: ONE layer of the benchmark workload solved by all ranks
    together (strong scaling): each rank accumulates the Hessian of its
    share of the tokens, one NCCL all-reduce sums S, rank 0 prepares U and
    broadcasts it with the order, and each rank quantizes and packs its own
    rows.  A step is one whole layer; the time is the max over ranks."""
    import torch
    from post_weight_quantization_31_b300 import api, build_lib, sharding
    build_lib.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    else:
        dist = _OneRank()
    inp = make_inputs()
    cfg = inp.cfg
    t0, t1 = sharding.token_range(N_TOK, world, rank)
    r0, r1 = sharding.row_range(D, world, rank)
    X_local = torch.from_numpy(np.ascontiguousarray(inp.X[:, t0:t1])).to(dev)
    W_rows = torch.from_numpy(inp.W[r0:r1]).to(torch.bfloat16).to(dev)
    S = torch.zeros((D, D), dtype=torch.float32, device=dev)
    U = torch.empty((D, D), dtype=torch.float32, device=dev)
    perm = torch.empty(D, dtype=torch.int32, device=dev)
    ws_prep = torch.empty(api.prepare_workspace_size(D), dtype=torch.uint8, device=dev)
    ws_q = torch.empty(api.quantize_workspace_size(r1 - r0, D, cfg), dtype=torch.uint8, device=dev)
    out = {}

    def prepare(S_, diag_, n, U_, perm_):
        api.prepare_hinv(S_, n, cfg, diag=diag_, U=U_, perm=perm_, ws=ws_prep, check=False)

    def quantize(Wr, U_, perm_):
        api.quantize_layer(Wr, U_, perm_, cfg, out=out, ws=ws_q, check=False)
        return api.pack(out["codes"], out["zeros"], cfg.bits, cfg.group_size)

    def step():
        S.zero_()
        sharding.sharded_layer_solve(dist, rank, X_local=X_local, W_rows=W_rows, rows=(r0, r1), S=S,
                                     diag=None, U=U, perm=perm,
                                     accumulate=lambda Xl, S_, d_: api.hessian_accumulate(Xl, S_, d_),
                                     prepare=prepare, quantize=quantize)

    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        clk.mark("start")
        a.record(stream)
        for _ in range(args.steps):
            step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        clk.mark("end")
    if rank == 0:
        api.workspace_status(ws_prep, "gptq_prepare_hinv")
    api.workspace_status(ws_q, "gptq_quantize_layer")
    ms = max_over_ranks(a.elapsed_time(b), dist if world > 1 else None, dev)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return None
    return {"metric": METRIC, "value": round(D * D * args.steps / (ms * 1e-3) / 1e6, 3),
            "unit": "Mweights/s", "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True, "scaling": "strong",
            "vs_baseline": None, "dtype": "fp16 x fp16 -> fp32 (Hessian), fp32 (solve)",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "d_row": D, "d_col": D, "n_tok": N_TOK,
                       "l2": "inputs larger than L2 (X is 2.15 GB)",
                       "parallelism": f"one layer: tokens and rows sharded over {world} GPU(s), "
                                      "all-reduce of S, broadcast of U"},
            "clocks": clk.summary()}


def measure_dequant(solver, cfg, stream, peaks: dict, reps: int) -> dict:
    """gptq_dequantize of the solved layer's packed output to fp16."""
    import torch
    return time_dequant(solver.qweight, solver.qzeros, solver.out["scales"], solver.out["g_idx"],
                        D, D, cfg.bits, cfg.group_size, torch.float16, stream, peaks, reps)


def time_dequant(qweight, qzeros, scales, g_idx, d_row, d_col, bits, group_size, dtype, stream,
                 peaks: dict, reps: int) -> dict:
    """Dequantization timed per launch with CUDA events on `stream`.  L2
    (126 MB) is flushed before each launch by reading a 256 MB buffer (a read
    leaves clean lines, so no write-back of earlier data lands inside the
    timed launch).  Algorithmic bytes: the packed words, zeros, scales and
    g_idx read once, the dense weights written once."""
    import torch
    from post_weight_quantization_31_b300 import api
    dev = qweight.device
    flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    out = torch.empty((d_row, d_col), dtype=dtype, device=dev)
    args = (qweight, qzeros, scales, g_idx, d_row, d_col, bits, group_size)
    for _ in range(2):
        api.dequantize(*args, dtype=dtype, out=out)
    ms = []
    for _ in range(reps):
        flush.sum()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        api.dequantize(*args, dtype=dtype, out=out)
        b.record(stream)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    nbytes = sum(t.numel() * t.element_size() for t in (qweight, qzeros, scales, g_idx, out))
    t = statistics.median(ms)
    gbs = nbytes / (t * 1e-3) / 1e9
    peak = float(peaks.get("hbm_gbs", 6400.0))
    tname = {torch.float16: "fp16", torch.bfloat16: "bf16", torch.float32: "fp32"}[dtype]
    return {"kernel": f"dequant_kernel ({d_row}x{d_col} {bits}-bit g{group_size} -> {tname})",
            "median_us": round(t * 1e3, 2), "bytes": int(nbytes), "reps": reps,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "peak_note": f"{peaks['source']} copy bandwidth"}}


def run_dequant_only(args) -> dict:
    """--dequant-only ROWSxCOLS: one packed 4-bit g128 layer (random codes,
    zeros and scales; packed by the library), dequantized to bf16."""
    import torch
    from post_weight_quantization_31_b300 import api, build_lib
    build_lib.build()
    d_row, d_col = (int(v) for v in args.dequant_only.lower().split("x"))
    bits, gs = 4, 128
    G = d_col // gs
    gen = torch.Generator(device="cuda").manual_seed(5)
    codes = torch.randint(0, 1 << bits, (d_row, d_col), dtype=torch.uint8, device="cuda", generator=gen)
    zeros = torch.randint(0, 1 << bits, (G, d_row), dtype=torch.uint8, device="cuda", generator=gen)
    qweight, qzeros = api.pack(codes, zeros, bits, gs)
    del codes
    scales = torch.rand((G, d_row), device="cuda", generator=gen) * 0.02 + 1e-3
    g_idx = (torch.arange(d_col, device="cuda", dtype=torch.int32) // gs).contiguous()
    res = time_dequant(qweight, qzeros, scales, g_idx, d_row, d_col, bits, gs, torch.bfloat16,
                       torch.cuda.current_stream(), measured_peaks(), max(1, args.dequant_reps))
    return {"metric": "dequantized weights GB/s (algorithmic bytes)", "value": res["roofline"]["achieved"],
            "unit": "GB/s", "n_gpus": 1, "higher_is_better": True, "data": "synthetic",
            "config": {"workload": f"packed {d_row}x{d_col} 4-bit g128 layer -> bf16, no act-order",
                       "l2": "flushed by a 256 MB read before each launch"},
            "dequant": res}


LAYER_SET_SITES = ("qkv", "o", "gate_up", "down")


def layer_set_inputs(dev) -> dict:
    """One decoder layer's inputs of the 7B-shaped layer set, on the device."""
    import torch
    from post_weight_quantization_31_b300 import api, workloads as wl
    sites = {}
    for site in LAYER_SET_SITES:
        inp = wl.decoder_site_7b(site, layer=0)
        d_row, d_col = inp.W.shape
        sites[site] = dict(X=torch.from_numpy(inp.X).to(dev),
                           W=torch.from_numpy(inp.W).to(torch.bfloat16).to(dev),
                           solver=api.LayerSolver(d_row, d_col, inp.cfg, device=dev), weights=d_row * d_col)
    return sites


def measure_layer_set(sites: dict, L: int, dev) -> dict:
    """L decoder layers x 4 input sites (q|k|v rows stacked on one X, o,
    gate|up stacked, down; 4-bit sym g128, 65536 tokens per site).  Each
    site: S = 0, accumulate, prepare, quantize, pack.  The inputs of one
    decoder layer are reused for every layer: each layer does the same work
    on data of the same distribution.
      sequential: one stream, layer after layer, site after site;
      concurrent: the four sites of each layer on four streams, enqueued
      round-robin from one host thread (every library call is asynchronous).
    Both are timed with CUDA events around the whole set; the device status
    of every solve is checked afterwards."""
    import torch
    weights_per_layer = sum(v["weights"] for v in sites.values())

    def solve(site):
        v = sites[site]
        v["solver"].reset()
        v["solver"].accumulate(v["X"])
        v["solver"].prepare()
        v["solver"].quantize(v["W"])
        v["solver"].pack()

    main = torch.cuda.current_stream(dev)
    for site in LAYER_SET_SITES:          # warm-up
        solve(site)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for _ in range(L):
        for site in LAYER_SET_SITES:
            solve(site)
    e1.record(main)
    torch.cuda.synchronize(dev)
    t_seq = e0.elapsed_time(e1) * 1e-3

    streams = {site: torch.cuda.Stream(dev) for site in LAYER_SET_SITES}
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    c0.record(main)
    for st in streams.values():
        st.wait_event(c0)
    for _ in range(L):
        for site in LAYER_SET_SITES:
            with torch.cuda.stream(streams[site]):
                solve(site)
    for st in streams.values():
        ev = torch.cuda.Event()
        ev.record(st)
        main.wait_event(ev)
    c1.record(main)
    torch.cuda.synchronize(dev)
    t_con = c0.elapsed_time(c1) * 1e-3
    for site in LAYER_SET_SITES:
        sites[site]["solver"].check()
    return {"sequential_s_per_32_layers": round(t_seq * 32 / L, 4),
            "concurrent_s_per_32_layers": round(t_con * 32 / L, 4),
            "layers_timed": L, "weights_per_layer": int(weights_per_layer),
            "sequential_mweights_s": round(weights_per_layer * L / t_seq / 1e6, 1),
            "concurrent_mweights_s": round(weights_per_layer * L / t_con / 1e6, 1),
            "workload": "32 x {q|k|v 12288x4096, o 4096x4096, gate|up 22016x4096, down 4096x11008} "
                        "bf16 N(0,0.02^2); X fp16 65536 tokens per site, N(0,1), 1% channels x "
                        "U[10,50]; 4-bit sym g128, damp 0.01, desc_act off; one decoder layer's "
                        "inputs reused for every layer"}


def run_layer_set(args) -> dict:
    """--layer-set L: the 7B-shaped layer set alone (see measure_layer_set)."""
    import torch
    from post_weight_quantization_31_b300 import build_lib
    build_lib.build()
    dev = torch.device("cuda", 0)
    r = measure_layer_set(layer_set_inputs(dev), int(args.layer_set), dev)
    return {"metric": "7B-shaped layer set: seconds per 32 decoder layers",
            "value": r["sequential_s_per_32_layers"], "unit": "s", "n_gpus": 1,
            "higher_is_better": False, "data": "synthetic",
            "config": {"workload": r["workload"], "layers_timed": r["layers_timed"]}, **r}


def run_awq(args) -> dict:
    """--awq: the AWQ scale search on the benchmark layer (4-bit g128, the 13
    candidates 1, 1.25, ..., 4, 5% salient channels).  A step: S = 0,
    accumulate (with the fp64 channel sums of squares the statistic needs),
    search (13 x: RTN of W diag(t), E = D S on the tensor cores, sum E .* D;
    then the choice and the final RTN on the device), pack.  Roofline: the
    search's GEMM flops (13 x 2 d_row d_col^2, useful products) against the
    measured 3xTF32 rate."""
    import torch
    from post_weight_quantization_31_b300 import api, build_lib
    build_lib.build()
    dev = torch.device("cuda", 0)
    inp = make_inputs()
    cfg = inp.cfg
    X = torch.from_numpy(inp.X).to(dev)
    W = torch.from_numpy(inp.W).to(torch.bfloat16).to(dev)
    S = torch.zeros((D, D), dtype=torch.float32, device=dev)
    diag = torch.zeros(D, dtype=torch.float64, device=dev)
    grid = api.AWQ_GRID
    ws = torch.empty(int(api._lib.load().gptq_awq_workspace_size(D, D, len(grid))), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]

    def step(e=None):
        S.zero_()
        diag.zero_()
        if e:
            e[0].record(stream)
        api.hessian_accumulate(X, S, diag)
        if e:
            e[1].record(stream)
        out = api.awq_search(W, S, diag, cfg, grid=grid, ws=ws, check=False)
        if e:
            e[2].record(stream)
        api.pack(out["codes"], out["zeros"], cfg.bits, cfg.group_size)
        if e:
            e[3].record(stream)
        return out

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    with ClockSampler(0) as clk:
        clk.mark("start")
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for k in range(args.steps):
            out = step(ev[k])
        t1.record(stream)
        torch.cuda.synchronize(dev)
        clk.mark("end")
    api.workspace_status(ws, "gptq_awq_search")
    ms = t0.elapsed_time(t1) / args.steps
    search_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    box = measure_box_peaks(dev)
    fl = len(grid) * 2.0 * D * D * D
    a = fl / (search_ms * 1e-3) / 1e12
    return {"metric": "AWQ layer search Mweights/s (4096x4096, 4-bit g128, 13 candidates)",
            "value": round(D * D / (ms * 1e-3) / 1e6, 3), "unit": "Mweights/s", "n_gpus": 1,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(ms, 4),
            "higher_is_better": True, "dtype": "fp16 x fp16 -> fp32 (Hessian), 3xTF32 / fp64 (errors)",
            "data": "synthetic",
            "config": {"workload": WORKLOAD.replace("desc_act off", "AWQ, 5% salient channels"),
                       "l2": "inputs larger than L2 (X is 2.15 GB)"},
            "phases_ms": {"hessian": round(statistics.mean(e[0].elapsed_time(e[1]) for e in ev), 4),
                          "search": round(search_ms, 4),
                          "pack": round(statistics.mean(e[2].elapsed_time(e[3]) for e in ev), 4)},
            "roofline": {"kernel": "tgemm_kernel (3xTF32, E = D S per candidate)", "bound": "tensor",
                         "achieved": round(a, 1), "peak": box["tf32x3_tflops"], "unit": "TFLOP/s",
                         "frac": round(a / box["tf32x3_tflops"], 4),
                         "peak_note": "measured cuBLAS TF32 / 3, this run; achieved over the whole search phase"},
            "chosen_factor": float(out["t"].max().item()),
            "clocks": clk.summary()}


def run_sweep(args) -> dict:
    """--sweep BITS:GS[:act],...: the bench step (S = 0, accumulate, prepare,
    quantize, pack) on the bench workload for other quantizer settings
    (group_size -1 = one group per row; act = desc_act on).  Timing as for
    the main line: W warm-up steps, then K steps between CUDA events."""
    import dataclasses

    import torch
    from post_weight_quantization_31_b300 import api, build_lib
    build_lib.build()
    dev = torch.device("cuda", 0)
    inp = make_inputs()
    X = torch.from_numpy(inp.X).to(dev)
    W = torch.from_numpy(inp.W).to(torch.bfloat16).to(dev)
    stream = torch.cuda.current_stream(dev)
    cases = []
    for spec in args.sweep.split(","):
        parts = spec.split(":")
        bits, gs = int(parts[0]), int(parts[1])
        act = len(parts) > 2 and parts[2] == "act"
        cfg = dataclasses.replace(inp.cfg, bits=bits, group_size=gs, desc_act=act)
        solver = api.LayerSolver(D, D, cfg, device=dev, exact_diag=False)

        def step():
            solver.reset()
            solver.accumulate(X)
            solver.prepare()
            solver.quantize(W)
            solver.pack()
        for _ in range(max(3, args.warmup)):
            step()
        torch.cuda.synchronize(dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        solver.check()
        ms = t0.elapsed_time(t1) / args.steps
        cases.append({"bits": bits, "group_size": gs, "desc_act": act, "ms_per_step": round(ms, 4),
                      "value": round(D * D / (ms * 1e-3) / 1e6, 3)})
        del solver
        torch.cuda.empty_cache()
    return {"metric": METRIC.split(" (")[0] + " (4096x4096, per quantizer setting)", "value": cases[0]["value"],
            "unit": "Mweights/s", "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup),
            "higher_is_better": True, "data": "synthetic",
            "config": {"workload": WORKLOAD.split("; 4-bit")[0] + "; settings per case",
                       "l2": "inputs larger than L2 (X is 2.15 GB)"},
            "cases": cases}


def run_dqgemm_only(args) -> dict:
    """--dqgemm-only MxNxK[,MxNxK...]: Y [M, N] = X [M, K] (fp16) times a
    random packed 4-bit g128 layer [N, K] (packed by the library),
    dequantized on the fly.  Algorithmic bytes: packed words, zeros, scales,
    g_idx and X read once, Y written once.  Each case also times cuBLAS
    (torch.matmul) on the same layer dequantized to dense fp16, for
    comparison."""
    import torch
    from post_weight_quantization_31_b300 import api, build_lib
    build_lib.build()
    peaks = measured_peaks()
    hbm, tc = float(peaks.get("hbm_gbs", 6400.0)), float(peaks.get("bf16_tflops", 1800.0))
    stream = torch.cuda.current_stream()
    flush = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
    reps = max(1, args.dequant_reps)

    def timed(fn):
        for _ in range(2):
            fn()
        ms = []
        for _ in range(reps):
            flush.sum()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        return statistics.median(ms)

    cases = []
    for shape in args.dqgemm_only.lower().split(","):
        M, N, K = (int(v) for v in shape.split("x"))
        bits, gs = 4, 128
        G = K // gs
        gen = torch.Generator(device="cuda").manual_seed(7)
        codes = torch.randint(0, 1 << bits, (N, K), dtype=torch.uint8, device="cuda", generator=gen)
        zeros = torch.randint(0, 1 << bits, (G, N), dtype=torch.uint8, device="cuda", generator=gen)
        qweight, qzeros = api.pack(codes, zeros, bits, gs)
        del codes
        scales = torch.rand((G, N), device="cuda", generator=gen) * 0.02 + 1e-3
        g_idx = (torch.arange(K, device="cuda", dtype=torch.int32) // gs).contiguous()
        X = torch.randn((M, K), device="cuda", generator=gen).half()
        Y = torch.empty((M, N), device="cuda")
        t = timed(lambda: api.dequant_matmul(X, qweight, qzeros, scales, g_idx, N, K, bits, gs, out=Y))
        case = {"M": M, "N": N, "K": K, "us": round(t * 1e3, 2)}
        if args.dqgemm_compare:
            Wd = api.dequantize(qweight, qzeros, scales, g_idx, N, K, bits, gs, dtype=torch.float16)
            case["cublas_dense_fp16_us"] = round(timed(lambda: torch.matmul(X, Wd.t())) * 1e3, 2)
            del Wd
        nbytes = sum(x.numel() * x.element_size() for x in (qweight, qzeros, scales, g_idx, X, Y))
        gbs = nbytes / (t * 1e-3) / 1e9
        tfl = 2.0 * M * N * K / (t * 1e-3) / 1e12
        case["roofline"] = {"hbm": {"achieved": round(gbs, 1), "frac": round(gbs / hbm, 4)},
                            "tensor": {"achieved": round(tfl, 1), "frac": round(tfl / tc, 4)}}
        cases.append(case)
        del qweight, qzeros, scales, X, Y
        torch.cuda.empty_cache()
    return {"metric": "fused dequant-GEMM time (us)", "value": cases[0]["us"], "unit": "us",
            "n_gpus": 1, "higher_is_better": False, "data": "synthetic", "reps": reps,
            "config": {"workload": "Y[M,N] = X[M,K] fp16 x packed 4-bit g128 W[N,K]^T, per case",
                       "l2": "flushed by a 256 MB read before each launch"},
            "peaks": {"hbm_gbs": hbm, "bf16_tflops": tc, "note": f"{peaks['source']} copy bandwidth and "
                                                                 "bf16 dense burst"},
            "cases": cases}


# ---------------------------------------------------------------- oracle arm
def _blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return int(max(n)) if n else 1
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(inp, quick: bool = False) -> dict:
    """Times the oracle on a bounded sample and extrapolates to one layer:
    Hessian on `tok` tokens (scaled by N/tok), the full prepare, the column
    loop and packing on `rows` rows (scaled by d_row/rows)."""
    import oracle as O
    tok = 2048 if quick else 8192
    rows = 16 if quick else 64
    t0 = time.perf_counter()
    S_s = O.hessian_sum(inp.X[:, :tok])
    t_h = time.perf_counter() - t0
    S_full = S_s * (N_TOK / tok)      # same scale as the full sum; values of the sample
    t0 = time.perf_counter()
    perm, Hp, U = O.prepare(S_full, N_TOK, inp.cfg)
    t_p = time.perf_counter() - t0
    t0 = time.perf_counter()
    Wp = inp.W[:rows].astype(np.float64)[:, perm]
    codes, scales, zeros, Q = O.column_loop(Wp, U, inp.cfg)
    t_q = time.perf_counter() - t0
    t0 = time.perf_counter()
    O.pack_qweight(codes, inp.cfg.bits)
    O.pack_qzeros(zeros, inp.cfg.bits)
    t_k = time.perf_counter() - t0
    full_s = t_h * (N_TOK / tok) + t_p + (t_q + t_k) * (D / rows)
    return {"value": round(D * D / full_s / 1e6, 6), "unit": "Mweights/s",
            "cores": _blas_threads(), "kind": "oracle",
            "sample": (f"Hessian on {tok} of {N_TOK} tokens (x{N_TOK // tok}), full prepare "
                       f"(d=4096), column loop + pack on {rows} of {D} rows (x{D // rows}); "
                       f"measured {t_h + t_p + t_q + t_k:.1f} s, extrapolated {full_s:.1f} s "
                       f"per layer"),
            "seconds_per_layer": round(full_s, 2)}


def run_reference(args, rank: int) -> dict | None:
    """The oracle as the reference arm.  The d^3 prepare is timed once; every
    step then times a small sample (Hessian on 1024 tokens, column loop and
    pack on 4 rows) and extrapolates one layer, so that --steps K stays
    within minutes for any K."""
    if rank != 0:
        return None
    import oracle as O
    inp = make_inputs()
    tok, rows = 1024, 8
    t0 = time.perf_counter()
    S_s = O.hessian_sum(inp.X[:, :tok])
    perm, _Hp, U = O.prepare(S_s * (N_TOK / tok), N_TOK, inp.cfg)
    t_prep = time.perf_counter() - t0
    secs = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        O.hessian_sum(inp.X[:, i * tok % N_TOK:][:, :tok])
        t_h = time.perf_counter() - t0
        r0 = (i * rows) % D
        t0 = time.perf_counter()
        Wp = inp.W[r0:r0 + rows].astype(np.float64)[:, perm]
        codes, _sc, zeros, _q = O.column_loop(Wp, U, inp.cfg)
        O.pack_qweight(codes, inp.cfg.bits)
        O.pack_qzeros(zeros, inp.cfg.bits)
        t_q = time.perf_counter() - t0
        if i >= args.warmup:
            secs.append(t_h * (N_TOK / tok) + t_prep + t_q * (D / rows))
    layer_s = statistics.median(secs)
    v = D * D / layer_s / 1e6
    sample = (f"per step: Hessian on {tok} of {N_TOK} tokens (x{N_TOK // tok}), column loop + pack "
              f"on {rows} of {D} rows (x{D // rows}); the full prepare (d=4096, {t_prep:.1f} s) "
              f"timed once and added; median over {args.steps} steps")
    return {"metric": METRIC, "value": round(v, 6), "unit": "Mweights/s", "impl": "reference",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(layer_s * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "d_row": D, "d_col": D, "n_tok": N_TOK},
            "cpu_baseline": {"value": round(v, 6), "unit": "Mweights/s", "cores": _blas_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 6), "unit": "Mweights/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--dequant-reps", type=int, default=20,
                    help="timed launches of the packed-layer dequantization (0: skip)")
    ap.add_argument("--dequant-only", default=None, metavar="ROWSxCOLS",
                    help="time only the dequantization of a packed layer of this shape")
    ap.add_argument("--layer-set", default=None, metavar="L",
                    help="time L decoder layers of the 7B-shaped layer set (sequential and concurrent)")
    ap.add_argument("--layer-set-layers", type=int, default=2,
                    help="decoder layers of the 7B-shaped layer set timed after the main line "
                         "(scaled to 32; 0: skip)")
    ap.add_argument("--sweep", default=None, metavar="BITS:GS[:act],...",
                    help="time the bench step for other quantizer settings")
    ap.add_argument("--dqgemm-only", default=None, metavar="MxNxK[,MxNxK...]",
                    help="time only the fused dequant-GEMM for these sizes")
    ap.add_argument("--dqgemm-compare", action="store_true",
                    help="with --dqgemm-only: also time cuBLAS on the dense fp16 weights")
    ap.add_argument("--awq", action="store_true", help="time the AWQ scale search on the benchmark layer")
    ap.add_argument("--shard", action="store_true",
                    help="solve one layer with all ranks together: token-sharded Hessian + "
                         "all-reduce, U broadcast, row-sharded quantize (strong scaling)")
    ap.add_argument("--quick-cpu", action="store_true", help="smaller oracle sample")
    ap.add_argument("--syrk-traffic", type=float, default=None,
                    help="DRAM bytes per Hessian launch from an ncu capture")
    ap.add_argument("--tokens", type=int, default=N_TOK,
                    help="calibration tokens (smaller values make a profiling case, "
                         "not the benchmark workload)")
    args = ap.parse_args()
    if args.tokens != N_TOK:
        set_tokens(args.tokens)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.dequant_only:
        line = run_dequant_only(args)
    elif args.dqgemm_only:
        line = run_dqgemm_only(args)
    elif args.sweep:
        line = run_sweep(args)
    elif args.layer_set:
        line = run_layer_set(args)
    elif args.awq:
        line = run_awq(args)
    elif args.shard and args.impl == "ours":
        line = run_sharded(args, rank, world, local_rank)
    elif args.impl == "reference":
        line = run_reference(args, rank)
    else:
        if args.warmup < 3:
            print("warning: fewer than 3 warm-up steps", file=sys.stderr)
        line = run_ours(args, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
