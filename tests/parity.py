"""Shared helpers for the GPU-vs-oracle parity tests.

Tolerances (the stated bar for the solver):
  scales within 1e-5 relative; >= 99.9% of codes identical and none more
  than 1 level apart; layer reconstruction error ||(W - Q) X||^2 within
  1e-3 relative; pack/unpack bit-exact.
"""
from __future__ import annotations

import dataclasses

import numpy as np

import oracle as O

SCALE_RTOL = 1e-5
CODE_MATCH = 0.999
RECON_RTOL = 1e-3


@dataclasses.dataclass
class GpuOut:
    codes: np.ndarray
    scales: np.ndarray
    zeros: np.ndarray
    g_idx: np.ndarray
    perm: np.ndarray
    U: np.ndarray
    S: np.ndarray
    diag: np.ndarray | None
    qweight: np.ndarray
    qzeros: np.ndarray
    n_seen: int


def torch_w(W: np.ndarray, w_dtype: str, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(W, dtype=np.float32))
    dt = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}[w_dtype]
    return t.to(dt).to(device)


def gpu_solve(W: np.ndarray, w_dtype: str, X: np.ndarray, cfg, chunks: int = 1,
              exact_diag: bool | None = None) -> GpuOut:
    import torch
    from post_weight_quantization_31_b300 import api
    d_row, d_col = W.shape
    Xd = torch.from_numpy(np.ascontiguousarray(X)).cuda()
    solver = api.LayerSolver(d_row, d_col, cfg, exact_diag=exact_diag)
    solver.reset()
    n = X.shape[1]
    bounds = np.linspace(0, n, chunks + 1).astype(int)
    for a, b in zip(bounds[:-1], bounds[1:]):
        if b > a:
            solver.accumulate(Xd[:, a:b].contiguous())
    solver.prepare()
    solver.quantize(torch_w(W, w_dtype))
    solver.pack()
    solver.check()
    torch.cuda.synchronize()
    o = solver.out
    return GpuOut(codes=o["codes"].cpu().numpy().astype(np.int64),
                  scales=o["scales"].cpu().numpy(), zeros=o["zeros"].cpu().numpy().astype(np.int64),
                  g_idx=o["g_idx"].cpu().numpy().astype(np.int64),
                  perm=solver.perm.cpu().numpy().astype(np.int64), U=solver.U.cpu().numpy(),
                  S=solver.S.cpu().numpy(),
                  diag=None if solver.diag is None else solver.diag.cpu().numpy(),
                  qweight=solver.qweight.cpu().numpy(), qzeros=solver.qzeros.cpu().numpy(),
                  n_seen=solver.n_seen)


def upstream_groups(g_codes, ref_codes, perm, group_size: int, n_groups: int) -> np.ndarray:
    """Mask [G, d_row] of the groups whose scale was set before the first code
    that differs in their row (in processing order).  A code decided on the
    other side of a rounding tie changes the compensation of every later
    column of its row, so later groups of that row legitimately differ."""
    diff = (g_codes != ref_codes)[:, perm]
    d_row, d_col = diff.shape
    first = np.where(diff.any(axis=1), diff.argmax(axis=1), d_col)
    if group_size == -1:
        return np.ones((n_groups, d_row), dtype=bool)
    gstart = np.arange(n_groups) * group_size
    return gstart[:, None] <= first[None, :]


# ---------------------------------------------------------------- measuring GPU outputs
# GPU outputs are measured with the plain NumPy below, never by passing them
# to the oracle: the oracle only ever sees the inputs.

def dequantized(codes, scales, zeros, g_idx) -> np.ndarray:
    """s[g][r] * (q[r][c] - z[g][r]) with g = g_idx[c], in fp64."""
    gi = np.asarray(g_idx, dtype=np.int64)
    s = np.asarray(scales, dtype=np.float64)[gi].T
    z = np.asarray(zeros, dtype=np.float64)[gi].T
    return s * (np.asarray(codes, dtype=np.float64) - z)


def output_error(W, Q, S64) -> float:
    """||(W - Q) X||^2 = tr(D S D^T) with S = X X^T (fp64)."""
    D = np.asarray(W, dtype=np.float64) - np.asarray(Q, dtype=np.float64)
    return float(np.einsum("ij,ij->", D @ np.asarray(S64, dtype=np.float64), D))


def unpack_columns(words, bits: int, count: int) -> np.ndarray:
    """Codes of each column of `words` (int32 [n_words, cols]): the column is
    one LSB-first bit stream of `count` codes of `bits` bits.  Returns
    int64 [cols, count]."""
    w = np.ascontiguousarray(np.asarray(words).T).astype("<u4")       # [cols, n_words]
    bitsarr = np.unpackbits(w.view(np.uint8), axis=1, bitorder="little")[:, :count * bits]
    weights = (1 << np.arange(bits, dtype=np.int64))
    return bitsarr.reshape(w.shape[0], count, bits).astype(np.int64) @ weights


def unpack_rows(words, bits: int, count: int) -> np.ndarray:
    """Codes of each row of `words` (int32 [rows, n_words]), LSB-first."""
    return unpack_columns(np.asarray(words).T, bits, count)


def compare(g: GpuOut, ref: O.LayerResult, W: np.ndarray, S64: np.ndarray, cfg) -> dict:
    """Metrics of a GPU result against the oracle's on the same inputs:
    codes, zeros, reconstruction error, and the scales of the groups
    upstream of any code difference.  The oracle only ever sees the inputs
    the GPU saw, never a GPU output."""
    same = g.codes == ref.codes
    eg = output_error(W, dequantized(g.codes, g.scales, g.zeros, g.g_idx), S64)
    er = O.recon_error(W, ref.Q, S64)
    rows_with_flip = int(np.any(~same, axis=1).sum())
    srel = np.abs(g.scales.astype(np.float64) - ref.scales) / np.abs(ref.scales.astype(np.float64))
    up = upstream_groups(g.codes, ref.codes, ref.perm, cfg.group_size, ref.scales.shape[0])
    m = dict(
        code_match=float(same.mean()),
        code_maxdiff=int(np.abs(g.codes - ref.codes).max()),
        zero_match=float((g.zeros == ref.zeros).mean()),
        zero_maxdiff=int(np.abs(g.zeros - ref.zeros).max()),
        scale_rel=float(srel[up].max()),
        scale_rel_all=float(srel.max()),
        upstream_frac=float(up.mean()),
        recon_gpu=eg, recon_ref=er, recon_rel=abs(eg - er) / er,
        rows_with_flip=rows_with_flip,
        perm_equal=bool(np.array_equal(g.perm, ref.perm)),
        g_idx_equal=bool(np.array_equal(g.g_idx, ref.g_idx)),
    )
    return m


def assert_parity(m: dict, scale_rtol: float = SCALE_RTOL) -> None:
    assert m["perm_equal"], m
    assert m["g_idx_equal"], m
    assert m["code_match"] >= CODE_MATCH, m
    assert m["code_maxdiff"] <= 1, m
    assert m["zero_match"] >= CODE_MATCH, m
    assert m["zero_maxdiff"] <= 1, m
    assert m["scale_rel"] <= scale_rtol, m
    assert m["recon_rel"] <= RECON_RTOL, m


def s_tol(n_tok: int) -> float:
    """Bound on max |dS_ij| / sqrt(S_ii S_jj) for fp32 sums of n_tok exact
    fp16 products: a random walk of ~n_tok/16 fp32 roundings (unit 6e-8)
    on partial sums up to sqrt(S_ii S_jj), with head-room (x8) for the
    maximum over up to 1e8 entries."""
    return 2e-7 * float(np.sqrt(n_tok)) + 2e-6


def s_error(S_gpu: np.ndarray, S64: np.ndarray) -> float:
    """max |dS_ij| / sqrt(S_ii S_jj)."""
    dg = np.sqrt(np.maximum(np.diag(S64), 1e-300))
    return float(np.max(np.abs(S_gpu.astype(np.float64) - S64) / np.outer(dg, dg)))
