"""CPU oracle of the AWQ scale search (activation-aware weight scaling).

TEST INFRASTRUCTURE ONLY, like the GPTQ oracle beside it: a plain NumPy fp64
restatement, imported only by the tests; no product code calls it.

Sources:
  [C]  "GPTQ/AWQ量化导出：让大模型在消费级显卡上跑起来", the GPTQ/AWQ comparison:
       AWQ takes the RMS of each channel's activations over the calibration
       data, picks the most active top-k% (5% by default), gives those
       channels a larger scale so they keep more effective bits, and
       multiplies back at inference.
  [E]  "大模型压缩量化技术：GPTQ 与 AWQ 原理详解 + Python 实战教程", §四 (AWQ
       原理): the weights of the large-activation channels are multiplied by a
       factor s > 1 before quantization, the matching activations are divided
       by s at inference so the output is unchanged, and the best factor is
       computed from forward statistics only (no Hessian inverse, no
       gradients).
  [S]  "AWQ与GPTQ谁更强？ms-swift量化模块深度评测", AWQ section: states the
       opposite direction (scale the non-salient channels down, leave the
       salient ones).  With a per-group min-max grid the two are the same
       relative scaling: a common factor on a whole row changes no code, so
       salient x s equals others x 1/s (pinned in the tests with s a power
       of two, where both are exact in floating point).

Readings (listed in the design notes as R17-R20):
  R17 statistic: RMS over the calibration tokens of each activation channel
      (W's input channel; [C] says "output channels", read as the
      channels of the activations that feed W, the ones divided by s).
  R18 salient set: the ceil(frac * d_col) channels with the largest RMS,
      frac = 0.05; ties keep the lower channel index.
  R19 factor: one factor s for the salient set, chosen on the grid
      1, 1.25, ..., 4 to minimise the layer output error ||(W - W_hat) X||^2
      = tr(D S D^T) with D = W - W_hat and S = X X^T; non-salient channels
      keep 1; ties take the smaller s, so s = 1 (plain round-to-nearest)
      wins unless scaling helps.
  R20 quantizer: the GPTQ oracle's round-to-nearest grid (its readings
      R6-R9), group-wise in natural column order, on W diag(t); the
      effective weights are W_hat = dequant / t, and at inference the
      activations are divided by t.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from .gptq_oracle import as_config, recon_error, rtn

SCALE_GRID = tuple(1.0 + 0.25 * i for i in range(13))     # 1, 1.25, ..., 4


@dataclass
class AwqResult:
    factor: float            # chosen s
    t: np.ndarray            # per-channel scale vector [d_col] (1 or s)
    salient: np.ndarray      # indices of the salient channels
    codes: np.ndarray        # codes of W diag(t)
    scales: np.ndarray
    zeros: np.ndarray
    W_hat: np.ndarray        # effective weights dequant / t
    error: float             # tr(D S D^T) at the chosen s
    errors: dict             # s -> error over the grid


def channel_rms(X: np.ndarray) -> np.ndarray:
    """RMS of each channel of X [d_col, n_tok] over its tokens (R17)."""
    X64 = np.asarray(X, dtype=np.float64)
    return np.sqrt(np.mean(X64 * X64, axis=1))


def salient_channels(rms: np.ndarray, frac: float = 0.05) -> np.ndarray:
    """The ceil(frac * d_col) channels with the largest RMS, ties to the
    lower index (R18); sorted ascending."""
    d = rms.shape[0]
    k = int(math.ceil(frac * d - 1e-12))
    order = np.lexsort((np.arange(d), -np.asarray(rms, dtype=np.float64)))
    return np.sort(order[:k])


def scaled_rtn(W: np.ndarray, t: np.ndarray, cfg):
    """Round-to-nearest of W diag(t) (R20); returns (codes, scales, zeros,
    W_hat) with W_hat = dequant / t."""
    W64 = np.asarray(W, dtype=np.float64)
    r = rtn(W64 * t[None, :], cfg)
    return r.codes, r.scales, r.zeros, r.Q / t[None, :]


def awq_search(W: np.ndarray, S: np.ndarray, rms: np.ndarray, cfg, frac: float = 0.05,
               grid=SCALE_GRID) -> AwqResult:
    """Search the salient channels' factor on `grid` (R18-R20)."""
    cfg = as_config(cfg)
    W64 = np.asarray(W, dtype=np.float64)
    sal = salient_channels(rms, frac)
    best = None
    errors = {}
    for s in grid:
        t = np.ones(W64.shape[1])
        t[sal] = s
        codes, scales, zeros, W_hat = scaled_rtn(W64, t, cfg)
        err = recon_error(W64, W_hat, S)
        errors[float(s)] = err
        if best is None or err < best.error:
            best = AwqResult(float(s), t, sal, codes, scales, zeros, W_hat, err, errors)
    best.errors = errors
    return best
