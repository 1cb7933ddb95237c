"""Seeded synthetic inputs for the GPTQ layer solver.

This module only draws random numbers in the shapes, sizes and value
distributions of the calibration workloads; it holds none of the solver's
arithmetic.  Tests feed the same bytes to the CUDA path and to the CPU oracle,
and the benchmark uses it to build its inputs.

Workload shapes follow the pages:
  * calibration set of 128 sequences x 2048 tokens (GPTQ practical guide,
    m.lqnn.cn/news/117696, §3.2 "选模型和校准数据") -> N = 262144 tokens;
  * 7B-shaped linear layers: q/k/v/o 4096x4096, gate/up 11008x4096,
    down 4096x11008; 13B-shaped: 5120x5120, 13824x5120, 5120x13824.
No dataset text is used: activations are drawn from N(0,1) with a few
large-magnitude "outlier" channels, or from a heavy-tailed Student-t.

All generators are deterministic functions of (seed, shape): the random
stream is split per block of channels with numpy's SeedSequence.spawn, so the
bytes do not depend on how many threads produce them.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

# Channels are generated in blocks of this many rows, each with its own
# child seed, so that generation can run on several threads.
_ROW_BLOCK = 64


@dataclasses.dataclass(frozen=True)
class QuantConfig:
    """The quantizer knobs of the pages (BaseQuantizeConfig / GptqConfig).

    bits, group_size, desc_act and damp_percent appear in the AutoGPTQ
    example of the GPTQ practical guide (m.lqnn.cn/news/117696, §3.3
    "量化超参怎么设置"); sym appears in the ms-swift GptqConfig example
    ("AWQ与GPTQ谁更强？ms-swift量化模块深度评测", GPTQ section); blocksize is
    the 128-column lazy batch (same guide, §2.2).
    """

    bits: int = 4
    group_size: int = 128
    damp_percent: float = 0.01
    blocksize: int = 128
    desc_act: bool = False
    sym: bool = False


@dataclasses.dataclass
class LayerInputs:
    """One linear layer's quantization problem.

    W: [d_row, d_col] (out_features x in_features), float32 values that are
       exactly representable in the stated storage dtype (bf16 or fp32).
    X: [d_col, n_tok] float16, channel-major (tokens contiguous).
    """

    name: str
    W: np.ndarray
    w_dtype: str  # "bf16" or "fp32"
    X: np.ndarray
    cfg: QuantConfig


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns
    float32 arrays whose values are bf16-representable."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) >> 16 << 16
    return u.astype(np.uint32).view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of bf16-representable float32 values."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def make_weight(d_row: int, d_col: int, seed: int, dtype: str = "bf16",
                std: float = 0.02) -> np.ndarray:
    """W ~ N(0, std^2), float32 then (for bf16) rounded to nearest bf16."""
    rng = np.random.Generator(np.random.PCG64(seed))
    w = rng.standard_normal((d_row, d_col), dtype=np.float32) * np.float32(std)
    if dtype == "bf16":
        w = round_to_bf16(w)
    elif dtype != "fp32":
        raise ValueError(dtype)
    return w


def _fill_rows(out: np.ndarray, seed: int, kind: str, nu: float) -> None:
    ss = np.random.SeedSequence(seed)
    n_blocks = (out.shape[0] + _ROW_BLOCK - 1) // _ROW_BLOCK
    children = ss.spawn(n_blocks)

    def work(b: int) -> None:
        rng = np.random.Generator(np.random.PCG64(children[b]))
        r0, r1 = b * _ROW_BLOCK, min(out.shape[0], (b + 1) * _ROW_BLOCK)
        if kind == "normal":
            blk = rng.standard_normal((r1 - r0, out.shape[1]), dtype=np.float32)
        else:
            blk = rng.standard_t(nu, size=(r1 - r0, out.shape[1])).astype(np.float32)
        out[r0:r1] = blk.astype(np.float16)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, range(n_blocks)))


def make_activations(d_col: int, n_tok: int, seed: int, *, kind: str = "normal",
                     outlier_frac: float = 0.0, n_outliers: int | None = None,
                     outlier_scale=(10.0, 50.0), nu: float = 4.0) -> np.ndarray:
    """Calibration activations X [d_col, n_tok] fp16 (channel-major).

    kind="normal": N(0,1); kind="student_t": Student-t with nu degrees of
    freedom, unscaled.  Outlier channels (a seeded random subset, either
    n_outliers of them or round(outlier_frac*d_col)) are multiplied by a
    per-channel factor: a fixed number if outlier_scale is a float, else
    uniform on the given interval.  Scaling is done in float32 before the
    cast to fp16.
    """
    X = np.empty((d_col, n_tok), dtype=np.float16)
    _fill_rows(X, seed, kind, nu)
    if n_outliers is None:
        n_outliers = int(round(outlier_frac * d_col))
    if n_outliers:
        rng = np.random.Generator(np.random.PCG64(seed ^ 0x5EED))
        chans = rng.permutation(d_col)[:n_outliers]
        if isinstance(outlier_scale, (int, float)):
            scales = np.full(n_outliers, float(outlier_scale), dtype=np.float32)
        else:
            lo, hi = outlier_scale
            scales = rng.uniform(lo, hi, size=n_outliers).astype(np.float32)
        for c, s in zip(chans, scales):
            X[c] = (X[c].astype(np.float32) * s).astype(np.float16)
    return X


def make_correlated_activations(d_col: int, n_tok: int, seed: int) -> np.ndarray:
    """X = A.Z with a seeded dense mixing matrix A (scaled so channels have
    unit variance) and Z ~ N(0,1).  Gives a strongly non-diagonal Hessian,
    where error compensation matters.  Small sizes only."""
    rng = np.random.Generator(np.random.PCG64(seed))
    A = rng.standard_normal((d_col, d_col)) / np.sqrt(d_col)
    A += np.eye(d_col) * 0.5
    Z = rng.standard_normal((d_col, n_tok))
    return (A @ Z).astype(np.float16)


def make_lowrank_activations(d_col: int, n_tok: int, seed: int, rank: int = 8,
                             noise: float = 0.1) -> np.ndarray:
    """Low-rank plus noise activations (small sizes only)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    B = rng.standard_normal((d_col, rank))
    C = rng.standard_normal((rank, n_tok))
    E = rng.standard_normal((d_col, n_tok)) * noise
    return (B @ C / np.sqrt(rank) + E).astype(np.float16)


# --------------------------------------------------------------------------
# The five calibration workloads.  `scale` divides the token count (and is
# used by tests to build reduced versions with the same distributions).
# --------------------------------------------------------------------------

CFG_TINY = QuantConfig(bits=4, group_size=128, damp_percent=0.01, blocksize=128,
                       desc_act=False, sym=False)
CFG_7B_ATTN = CFG_TINY
CFG_7B_MLP = QuantConfig(bits=4, group_size=128, damp_percent=0.01, blocksize=128,
                         desc_act=True, sym=False)
CFG_7B_SET = QuantConfig(bits=4, group_size=128, damp_percent=0.01, blocksize=128,
                         desc_act=False, sym=True)


def cfg_13b_lowbit(bits: int) -> QuantConfig:
    return QuantConfig(bits=bits, group_size=64, damp_percent=0.1, blocksize=128,
                       desc_act=True, sym=True)


def tiny_layer(seed: int = 1001) -> LayerInputs:
    """256x512 fp32 W; X 512x2048 N(0,1) with 8 outlier channels x20."""
    W = make_weight(256, 512, seed, dtype="fp32")
    X = make_activations(512, 2048, seed + 1, n_outliers=8, outlier_scale=20.0)
    return LayerInputs("tiny_256x512", W, "fp32", X, CFG_TINY)


def attn_proj_7b(seed: int = 1002, n_tok: int = 262144, d: int = 4096) -> LayerInputs:
    """4096x4096 bf16 W; X 4096 x 262144 N(0,1), 1% channels x U[10,50]."""
    W = make_weight(d, d, seed, dtype="bf16")
    X = make_activations(d, n_tok, seed + 1, outlier_frac=0.01,
                         outlier_scale=(10.0, 50.0))
    return LayerInputs(f"attn_proj_{d}x{d}_N{n_tok}", W, "bf16", X, CFG_7B_ATTN)


def mlp_7b(which: str, seed: int = 1003, n_tok: int = 262144,
           d_model: int = 4096, d_ff: int = 11008) -> LayerInputs:
    """gate|up (d_ff x d_model, sharing one X) or down (d_model x d_ff);
    X heavy-tailed Student-t nu=4; desc_act on."""
    if which == "gate_up":
        W = make_weight(2 * d_ff, d_model, seed, dtype="bf16")
        X = make_activations(d_model, n_tok, seed + 1, kind="student_t", nu=4.0)
    elif which == "down":
        W = make_weight(d_model, d_ff, seed + 10, dtype="bf16")
        X = make_activations(d_ff, n_tok, seed + 11, kind="student_t", nu=4.0)
    else:
        raise ValueError(which)
    return LayerInputs(f"mlp_{which}", W, "bf16", X, CFG_7B_MLP)


def decoder_site_7b(site: str, layer: int = 0, n_tok: int = 65536) -> LayerInputs:
    """One input site of a 7B-shaped decoder layer (the 32-layer set): the
    matrices that read the same activations share one X, so their rows are
    stacked into one W.  site: "qkv" (3 x 4096 rows, d_col 4096), "o"
    (4096 x 4096), "gate_up" (2 x 11008 rows, d_col 4096), "down"
    (4096 x 11008).  X: N(0,1) with 1% of channels x U[10,50]; 4-bit sym g128."""
    shapes = {"qkv": (3 * 4096, 4096), "o": (4096, 4096), "gate_up": (2 * 11008, 4096),
              "down": (4096, 11008)}
    d_row, d_col = shapes[site]
    seed = 1004 + 100 * layer + {"qkv": 0, "o": 10, "gate_up": 20, "down": 30}[site]
    W = make_weight(d_row, d_col, seed, dtype="bf16")
    X = make_activations(d_col, n_tok, seed + 1, outlier_frac=0.01, outlier_scale=(10.0, 50.0))
    return LayerInputs(f"decoder{layer}_{site}", W, "bf16", X, CFG_7B_SET)


def lowbit_13b(which: str, bits: int, n_tok: int = 131072) -> LayerInputs:
    """13B-shaped low-bit sweep: "attn" 5120x5120, "gate_up" 2 x 13824 rows
    x 5120 (one shared X), "down" 5120 x 13824.  X: N(0,1) with 1% of
    channels x U[10,50]; bits 3 or 2, sym, g64, damp 0.1, desc_act on."""
    shapes = {"attn": (5120, 5120), "gate_up": (2 * 13824, 5120), "down": (5120, 13824)}
    d_row, d_col = shapes[which]
    seed = 1005 + {"attn": 0, "gate_up": 10, "down": 20}[which]
    W = make_weight(d_row, d_col, seed, dtype="bf16")
    X = make_activations(d_col, n_tok, seed + 1, outlier_frac=0.01, outlier_scale=(10.0, 50.0))
    return LayerInputs(f"lowbit13b_{which}_{bits}bit", W, "bf16", X, cfg_13b_lowbit(bits))
