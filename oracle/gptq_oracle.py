"""CPU oracle of the GPTQ per-layer quantization solver.

TEST INFRASTRUCTURE ONLY.  This module is a plain, slow, obviously-correct
NumPy restatement of what the solver computes.  It is imported only by the
tests, by the package's smoke check and by the benchmark's CPU-baseline leg;
the product path never calls it, and it shares no code with the CUDA library.

Sources (the web pages this method is described on):
  [G]  GPTQ practical guide, m.lqnn.cn/news/117696
       §2.1 "从OBQ说起" (OBQ update), §2.2 "固定顺序、Lazy Batch、Cholesky",
       §3.3 "量化超参怎么设置" (bits, group_size, desc_act, damp_percent),
       §5.2 (desc_act column re-order at load time).
  [E]  "大模型压缩量化技术：GPTQ 与 AWQ 原理详解 + Python 实战教程",
       §二 (min-max round-to-nearest), §三 (quantize one, compensate the rest),
       FAQ Q6 (group_size, -1 = one group per row).
  [S]  "AWQ与GPTQ谁更强？ms-swift量化模块深度评测", GPTQ section
       (GptqConfig(..., damp_percent=0.01, desc_act, sym=True)).

Precision: everything is fp64 -- H, U, the weights during the column loop,
the errors, and the quantizer decisions.  The one fp32 number is the
group's scale: it is stored as fp32 (the output type of the scales), and the
zero point and every code are decided against that stored value with the
plain definitions, z = rint(-xmin / s) and code = clamp(rint(w / s) + z, 0,
maxq), so that the grid the codes were chosen on is the grid s * (q - z)
that dequantization rebuilds.

Readings taken where the pages are silent or garbled (each listed in the
design notes):
  R1 (§2.1 formula is printed without quant()): the update is
     delta_F = -(w_q - quant(w_q)) / [Hinv]_qq * Hinv[:, q] on the
     not-yet-quantized weights F.
  R2 (order): desc_act off -> natural order; on -> descending diag(H) with a
     stable sort (ties keep the lower original index first), processed first
     to last.
  R3 (H scale): S = X X^T is accumulated unnormalized; H = (2/n) S.
  R4 (damping): lambda = damp_percent * mean(diag H), added to diag(H).
  R5 (which values set a group's scale): the current, error-updated values of
     the group's columns when the loop reaches the group's first column
     (group_size = -1: the initial row, before any update).
  R6 (asymmetric range): [min(0, min w), max(0, max w)], so the zero point is
     a valid unsigned code.
  R7 (symmetric): a = max(|xmin|, xmax), s = 2a/maxq, z = (maxq+1)/2.
  R8 (degenerate range xmin == xmax): use [-1, +1].
  R9 (rounding): round half to even, applied to the exact quotient w / s
     (here evaluated in fp64).
  R10 (groups under desc_act): gs consecutive columns in processing order;
      g_idx maps each original column to its group.
  R11 (packing, not on the pages): LSB-first along the input dimension;
      3-bit packs 32 codes into 3 words as one bit stream.
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass(frozen=True)
class OracleConfig:
    bits: int = 4
    group_size: int = 128
    damp_percent: float = 0.01
    blocksize: int = 128
    desc_act: bool = False
    sym: bool = False


def as_config(cfg) -> OracleConfig:
    """Accept any object with the six knob attributes."""
    return OracleConfig(bits=int(cfg.bits), group_size=int(cfg.group_size),
                        damp_percent=float(cfg.damp_percent),
                        blocksize=int(cfg.blocksize), desc_act=bool(cfg.desc_act),
                        sym=bool(cfg.sym))


# --------------------------------------------------------------------------
# a1: Hessian.  [G] §2.1: H is built from the layer's calibration
# activations; the standard form is H = 2/N * X X^T (R3).
# --------------------------------------------------------------------------

def hessian_sum(X: np.ndarray) -> np.ndarray:
    """S = X X^T in fp64 for X [d_col, n_tok] (fp16 values are exact in fp64)."""
    X64 = np.asarray(X, dtype=np.float64)
    return X64 @ X64.T


def hessian_sum_chunked(X: np.ndarray, chunk: int = 16384) -> np.ndarray:
    """The same S = X X^T in fp64, summed over chunks of tokens so that the
    fp64 copy of X never has to exist whole (full-size layers)."""
    d = X.shape[0]
    S = np.zeros((d, d), dtype=np.float64)
    for t0 in range(0, X.shape[1], chunk):
        Xc = np.asarray(X[:, t0:t0 + chunk], dtype=np.float64)
        S += Xc @ Xc.T
    return S


def hessian_diag(X: np.ndarray, chunk: int = 16384) -> np.ndarray:
    """diag(S) = sum_t X[i, t]^2 in fp64, by token chunks."""
    out = np.zeros(X.shape[0], dtype=np.float64)
    for t0 in range(0, X.shape[1], chunk):
        Xc = np.asarray(X[:, t0:t0 + chunk], dtype=np.float64)
        out += np.einsum("ij,ij->i", Xc, Xc)
    return out


def hessian_columns(X: np.ndarray, cols, chunk: int = 8192) -> np.ndarray:
    """Columns S[:, cols] = X X[cols]^T in fp64, by token chunks."""
    cols = np.asarray(cols)
    out = np.zeros((X.shape[0], len(cols)), dtype=np.float64)
    for t0 in range(0, X.shape[1], chunk):
        Xc = np.asarray(X[:, t0:t0 + chunk], dtype=np.float64)
        out += Xc @ Xc[cols].T
    return out


def hessian_entry(X: np.ndarray, i: int, j: int) -> float:
    """One entry S[i, j] = sum_t X[i, t] X[j, t], computed on its own."""
    xi = np.asarray(X[i], dtype=np.float64)
    xj = np.asarray(X[j], dtype=np.float64)
    return float(np.dot(xi, xj))


# --------------------------------------------------------------------------
# a2: damping, column order, Cholesky factor of H^-1.
# --------------------------------------------------------------------------

def damped_hessian(S: np.ndarray, n_seen: int, damp_percent: float) -> np.ndarray:
    """H = (2/n) S + lambda I, lambda = damp_percent * mean(diag H).

    [G] §3.3 (damp_percent adds a small damping to the Hessian diagonal to
    avoid a singular matrix); [S] (damp_percent=0.01 "防止Hessian奇异").
    """
    H = (2.0 / float(n_seen)) * np.asarray(S, dtype=np.float64)
    lam = float(damp_percent) * float(np.mean(np.diag(H)))
    return H + lam * np.eye(H.shape[0])


def act_order(H: np.ndarray, desc_act: bool) -> np.ndarray:
    """Processing order (R2).  [G] §2.2: columns are ordered once, up front,
    by the Hessian diagonal from large to small; §3.3: desc_act switches it.
    Stable sort: equal diagonals keep their original relative order."""
    return act_order_diag(np.diag(H), desc_act)


def act_order_diag(hdiag: np.ndarray, desc_act: bool) -> np.ndarray:
    """act_order from the Hessian diagonal alone."""
    n = len(hdiag)
    if not desc_act:
        return np.arange(n, dtype=np.int64)
    return np.argsort(-np.asarray(hdiag, dtype=np.float64), kind="stable").astype(np.int64)


def hinv_upper(H: np.ndarray) -> np.ndarray:
    """Upper-triangular U with H^-1 = U^T U and U_ii > 0.

    [G] §2.2 ("第三，用Cholesky分解简化计算"): the inverse Hessian is used
    through a Cholesky factor.  Textbook chain: L = chol(H),
    H^-1 = L^-T L^-1, U = chol(H^-1)^T.  Raises numpy's LinAlgError when H
    is not positive definite.
    """
    L = np.linalg.cholesky(H)
    Linv = np.linalg.inv(L)
    Hinv = Linv.T @ Linv
    Hinv = 0.5 * (Hinv + Hinv.T)
    return np.linalg.cholesky(Hinv).T


def hinv_upper_reverse(H: np.ndarray) -> np.ndarray:
    """The same U by the other route: H = R R^T with R upper (a Cholesky
    factorization taken from the last index to the first), then U = R^-1.
    Written out element by element on purpose (small n only)."""
    n = H.shape[0]
    A = np.array(H, dtype=np.float64)
    R = np.zeros_like(A)
    for j in range(n - 1, -1, -1):
        piv = A[j, j] - np.dot(R[j, j + 1:], R[j, j + 1:])
        if not piv > 0:
            raise np.linalg.LinAlgError("not positive definite")
        R[j, j] = np.sqrt(piv)
        for i in range(j - 1, -1, -1):
            R[i, j] = (A[i, j] - np.dot(R[i, j + 1:], R[j, j + 1:])) / R[j, j]
    # Back substitution for the inverse of the upper-triangular R.
    U = np.zeros_like(R)
    for j in range(n):
        U[j, j] = 1.0 / R[j, j]
        for i in range(j - 1, -1, -1):
            U[i, j] = -np.dot(R[i, i + 1:j + 1], U[i + 1:j + 1, j]) / R[i, i]
    return U


def prepare(S: np.ndarray, n_seen: int, cfg) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """a2 in full: returns (perm, Hp, U) where Hp = H[perm][:, perm] is the
    damped Hessian in processing order and U its inverse Cholesky factor.
    perm[i] is the original index of the column processed i-th."""
    cfg = as_config(cfg)
    H = damped_hessian(S, n_seen, cfg.damp_percent)
    perm = act_order(H, cfg.desc_act)
    Hp = H[np.ix_(perm, perm)]
    return perm, Hp, hinv_upper(Hp)


# --------------------------------------------------------------------------
# The quantizer grid.  [E] §二: min-max uniform quantization, each weight
# rounded to the nearest level; [G] §3.3: one scale and zero point per
# group_size consecutive columns; [S]: sym=True selects the symmetric grid.
# --------------------------------------------------------------------------

def maxq_of(bits: int) -> int:
    return (1 << int(bits)) - 1


def quant_params(w: np.ndarray, bits: int, sym: bool, include_zero: bool = True):
    """Grid of each row of w [rows, g] (R6-R8), from the fp64 values.

    Asymmetric: xmin = min(0, min w), xmax = max(0, max w) (R6), span =
    xmax - xmin, s = span / maxq, z = rint(-xmin / s).  Symmetric (R7):
    a = max(|xmin|, xmax), span = 2a, s = 2a / maxq, z = (maxq + 1) / 2.  An
    empty range (xmin == xmax, or a == 0) uses [-1, 1] instead (R8).

    Returns (scale float32 [rows], zero int64 [rows], span float64 [rows]).
    The scale is stored as fp32, the output type; decisions (the zero point
    here, the codes in quantize_codes) are taken on the exact quotient
    x / s = maxq * (x / span), not on the stored fp32 scale (R9).
    include_zero=False gives the unconstrained min-max grid of the pages'
    worked example (the zero point may then fall outside [0, maxq]); the
    solver always uses include_zero=True.
    """
    maxq = maxq_of(bits)
    w64 = np.asarray(w, dtype=np.float64)
    xmin = w64.min(axis=1)
    xmax = w64.max(axis=1)
    if include_zero:
        xmin = np.minimum(xmin, 0.0)
        xmax = np.maximum(xmax, 0.0)
    if sym:
        a = np.maximum(np.abs(xmin), xmax)
        a = np.where(a == 0, 1.0, a)
        span = 2.0 * a
        zero = np.full(w64.shape[0], (maxq + 1) // 2, dtype=np.int64)
    else:
        deg = xmin == xmax
        xmin = np.where(deg, -1.0, xmin)
        xmax = np.where(deg, 1.0, xmax)
        span = xmax - xmin
        zero = np.rint(maxq * (-xmin / span)).astype(np.int64)
    scale = (span / maxq).astype(np.float32)
    return scale, zero, span


def quantize_codes(w: np.ndarray, span: np.ndarray, zero: np.ndarray, bits: int) -> np.ndarray:
    """code = clamp(rint(w / s) + z, 0, maxq) with s = span / maxq (R9),
    evaluated in fp64 as rint(maxq * (w / span)), half to even.  Written this
    way, a weight exactly at a grid midpoint (such as -a on the symmetric
    grid, which lands on -maxq/2) gives an exact midpoint here too."""
    maxq = maxq_of(bits)
    t = np.rint(maxq * (np.asarray(w, dtype=np.float64) / np.asarray(span, dtype=np.float64)))
    return np.clip(t.astype(np.int64) + zero, 0, maxq)


def dequantize_codes(q: np.ndarray, scale: np.ndarray, zero: np.ndarray) -> np.ndarray:
    """dq = s (q - z) in fp64 (s is the fp32 scale)."""
    return np.asarray(scale, dtype=np.float64) * (np.asarray(q, dtype=np.float64) - zero)


# --------------------------------------------------------------------------
# a3 + a4: the column loop with OBQ error feedback and lazy batch updates.
# --------------------------------------------------------------------------

def obq_error(w: np.ndarray, dq: np.ndarray, u_jj: float) -> np.ndarray:
    """e = (w_j - quant(w_j)) / U_jj, the scaled quantization error of column j."""
    return (w - dq) / u_jj


def obq_update(W: np.ndarray, e: np.ndarray, U: np.ndarray, j: int, k1: int, k2: int) -> None:
    """W[:, k1:k2] -= e U[j, k1:k2]: the OBQ compensation ([G] §2.1, R1)
    applied to columns k1..k2-1 of the current block."""
    W[:, k1:k2] -= np.outer(e, U[j, k1:k2])


def lazy_trailing_update(W: np.ndarray, Err: np.ndarray, U: np.ndarray, i1: int, i2: int) -> None:
    """W[:, i2:] -= Err U[i1:i2, i2:]: one matrix multiply for all columns
    after the block ([G] §2.2, Lazy Batch-Updates)."""
    W[:, i2:] -= Err @ U[i1:i2, i2:]


def _check_blocking(d_col: int, gs: int, blocksize: int) -> None:
    if gs != -1:
        if gs <= 0 or d_col % gs:
            raise ValueError("group_size must divide d_col (or be -1)")
        if blocksize % gs and gs % blocksize:
            raise ValueError("group starts must coincide with block starts")


def column_loop(Wp: np.ndarray, U: np.ndarray, cfg, *, blocksize: int | None = None, trace=None):
    """Quantize Wp [rows, d_col] (processing order, fp64) with error feedback.

    For each block [i1, i2) of `blocksize` columns, for j in the block, per
    row ([G] §2.1 OBQ step with R1, rewritten through the Cholesky factor:
    row q of the inverse Hessian restricted to the unquantized set equals
    U_qq * U[q, q:], so the update is w_F -= (w_q - dq)/U_qq * U[q, F]):
      at a group start, (scale, zero) from the current W[:, j:j+gs] (R5);
      q  = code(w_j);  dq = s (q - z);  e = (w_j - dq) / U_jj;
      W[:, j+1:i2] -= e U[j, j+1:i2];  Err[:, j-i1] = e.
    After the block ([G] §2.2 lazy batch: quantize 128 columns, then update
    all remaining weights with one matrix multiply):
      W[:, i2:] -= Err U[i1:i2, i2:].

    trace(j, W) is called after column j's in-block update (and, at a
    block end, after the trailing update).

    Returns codes int64 [rows, d_col], scales float32 [G, rows],
    zeros int64 [G, rows], Q float64 [rows, d_col] (dequantized values), all
    in processing order.
    """
    cfg = as_config(cfg)
    W = np.array(Wp, dtype=np.float64)
    rows, d_col = W.shape
    B = int(blocksize if blocksize is not None else cfg.blocksize)
    gs = cfg.group_size
    _check_blocking(d_col, gs, B)
    n_groups = 1 if gs == -1 else d_col // gs
    scales = np.zeros((n_groups, rows), dtype=np.float32)
    zeros = np.zeros((n_groups, rows), dtype=np.int64)
    codes = np.zeros((rows, d_col), dtype=np.int64)
    Q = np.zeros((rows, d_col), dtype=np.float64)
    spans = np.zeros((n_groups, rows), dtype=np.float64)
    if gs == -1:
        scales[0], zeros[0], spans[0] = quant_params(W, cfg.bits, cfg.sym)
    s, z, sp = scales[0].copy(), zeros[0].copy(), spans[0].copy()
    for i1 in range(0, d_col, B):
        i2 = min(i1 + B, d_col)
        Err = np.zeros((rows, i2 - i1), dtype=np.float64)
        for j in range(i1, i2):
            if gs != -1 and j % gs == 0:
                g = j // gs
                scales[g], zeros[g], spans[g] = quant_params(W[:, j:j + gs], cfg.bits, cfg.sym)
                s, z, sp = scales[g].copy(), zeros[g].copy(), spans[g].copy()
            w = W[:, j]
            q = quantize_codes(w, sp, z, cfg.bits)
            dq = dequantize_codes(q, s, z)
            e = obq_error(w, dq, U[j, j])
            obq_update(W, e, U, j, j + 1, i2)
            Err[:, j - i1] = e
            codes[:, j] = q
            Q[:, j] = dq
            if trace is not None and j + 1 < i2:
                trace(j, W)
        if i2 < d_col:
            lazy_trailing_update(W, Err, U, i1, i2)
        if trace is not None:
            trace(i2 - 1, W)
    return codes, scales, zeros, Q


def group_index(perm: np.ndarray, group_size: int) -> np.ndarray:
    """g_idx[perm[i]] = i // gs: the group of each ORIGINAL column (R10;
    [G] §5.2, columns are re-ordered back at load/inference time)."""
    d_col = perm.shape[0]
    g_idx = np.zeros(d_col, dtype=np.int64)
    if group_size == -1:
        return g_idx
    g_idx[perm] = np.arange(d_col) // group_size
    return g_idx


@dataclasses.dataclass
class LayerResult:
    codes: np.ndarray      # int64 [d_row, d_col], ORIGINAL column order
    scales: np.ndarray     # float32 [G, d_row]
    zeros: np.ndarray      # int64 [G, d_row]
    g_idx: np.ndarray      # int64 [d_col]
    perm: np.ndarray       # int64 [d_col], processing position -> original column
    Q: np.ndarray          # float64 [d_row, d_col] dequantized weights, original order
    U: np.ndarray | None = None


def quantize_layer(W: np.ndarray, S: np.ndarray, n_seen: int, cfg, *,
                   blocksize: int | None = None, rows=None) -> LayerResult:
    """The whole solve for one layer (a2 .. a5 minus packing).

    W [d_row, d_col] holds the layer's weights (bf16/fp32 values, used in
    fp64).  `rows` restricts the solve to a subset of rows (rows are
    independent).
    """
    cfg = as_config(cfg)
    perm, _Hp, U = prepare(S, n_seen, cfg)
    W64 = np.asarray(W, dtype=np.float64)
    if rows is not None:
        W64 = W64[np.asarray(rows)]
    Wp = W64[:, perm]
    codes_p, scales, zeros, Q_p = column_loop(Wp, U, cfg, blocksize=blocksize)
    codes = np.empty_like(codes_p)
    Q = np.empty_like(Q_p)
    codes[:, perm] = codes_p
    Q[:, perm] = Q_p
    return LayerResult(codes=codes, scales=scales, zeros=zeros,
                       g_idx=group_index(perm, cfg.group_size), perm=perm, Q=Q, U=U)


def rtn(W: np.ndarray, cfg) -> LayerResult:
    """Round-to-nearest baseline ([E] §二): the same grid, natural order,
    no error compensation."""
    cfg = as_config(cfg)
    W64 = np.asarray(W, dtype=np.float64)
    d_row, d_col = W64.shape
    gs = cfg.group_size
    n_groups = 1 if gs == -1 else d_col // gs
    width = d_col if gs == -1 else gs
    scales = np.zeros((n_groups, d_row), dtype=np.float32)
    zeros = np.zeros((n_groups, d_row), dtype=np.int64)
    codes = np.zeros((d_row, d_col), dtype=np.int64)
    Q = np.zeros((d_row, d_col))
    for g in range(n_groups):
        blk = W64[:, g * width:(g + 1) * width]
        scales[g], zeros[g], span = quant_params(blk, cfg.bits, cfg.sym)
        q = quantize_codes(blk, span[:, None], zeros[g][:, None], cfg.bits)
        codes[:, g * width:(g + 1) * width] = q
        Q[:, g * width:(g + 1) * width] = dequantize_codes(q, scales[g][:, None],
                                                          zeros[g][:, None])
    perm = np.arange(d_col, dtype=np.int64)
    return LayerResult(codes=codes, scales=scales, zeros=zeros,
                       g_idx=group_index(perm, gs), perm=perm, Q=Q)


def dequantize(codes: np.ndarray, scales: np.ndarray, zeros: np.ndarray,
               g_idx: np.ndarray) -> np.ndarray:
    """W_hat[r, c] = scales[g_idx[c], r] * (codes[r, c] - zeros[g_idx[c], r])."""
    s = np.asarray(scales, dtype=np.float64)[g_idx].T
    z = np.asarray(zeros, dtype=np.float64)[g_idx].T
    return s * (np.asarray(codes, dtype=np.float64) - z)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 values rounded to the nearest bfloat16 (ties to even), returned
    as float32: keep the top 16 bits after adding half an ulp of bf16."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32)


def dequantize_as(codes: np.ndarray, scales: np.ndarray, zeros: np.ndarray, g_idx: np.ndarray,
                  dtype: str) -> np.ndarray:
    """Dense weights as stored in `dtype` ("fp32", "fp16", "bf16"): the
    product scale * (code - zero) formed in fp32 (the difference is a small
    exact integer), then rounded to nearest in the storage type."""
    s = np.asarray(scales, dtype=np.float32)[g_idx].T
    dq = (np.asarray(codes, dtype=np.int64) - np.asarray(zeros, dtype=np.int64)[g_idx].T).astype(np.float32)
    w = (s * dq).astype(np.float32)
    if dtype == "fp32":
        return w
    if dtype == "fp16":
        return w.astype(np.float16).astype(np.float32)
    if dtype == "bf16":
        return round_bf16(w)
    raise ValueError(dtype)


def dequant_matmul(X: np.ndarray, codes: np.ndarray, scales: np.ndarray, zeros: np.ndarray,
                   g_idx: np.ndarray, dtype: str) -> np.ndarray:
    """Y = X · Wᵀ in fp64, W the dequantized layer as stored in `dtype`
    ([G] §4.3: the codes are unpacked to 16-bit weights, then multiplied).
    X holds the values of the 16-bit activations."""
    W = dequantize_as(codes, scales, zeros, g_idx, dtype).astype(np.float64)
    return np.asarray(X, dtype=np.float64) @ W.T


def recon_error(W: np.ndarray, Q: np.ndarray, S: np.ndarray) -> float:
    """||(W - Q) X||_F^2 = tr((W - Q) S (W - Q)^T) with the undamped S = X X^T."""
    D = np.asarray(W, dtype=np.float64) - np.asarray(Q, dtype=np.float64)
    return float(np.einsum("ij,ij->", D @ np.asarray(S, dtype=np.float64), D))


# --------------------------------------------------------------------------
# a5: packing into int32 words (R11).  Pure-Python integer bit operations,
# one word at a time: small inputs only.
# --------------------------------------------------------------------------

def _pack_stream(vals, bits: int) -> list[int]:
    """LSB-first bit stream of `vals` cut into 32-bit words."""
    acc, nacc, out = 0, 0, []
    for v in vals:
        v = int(v)
        if not 0 <= v < (1 << bits):
            raise ValueError("code out of range")
        acc |= v << nacc
        nacc += bits
        while nacc >= 32:
            out.append(acc & 0xFFFFFFFF)
            acc >>= 32
            nacc -= 32
    if nacc:
        raise ValueError("stream length is not a whole number of words")
    return out


def _unpack_stream(words, bits: int, count: int) -> list[int]:
    acc, nacc, out = 0, 0, []
    it = iter(words)
    mask = (1 << bits) - 1
    while len(out) < count:
        if nacc < bits:
            acc |= (int(next(it)) & 0xFFFFFFFF) << nacc
            nacc += 32
        out.append(acc & mask)
        acc >>= bits
        nacc -= bits
    return out


def _as_i32(words: list[int]) -> np.ndarray:
    return np.array(words, dtype=np.uint64).astype(np.uint32).view(np.int32)


def pack_qweight(codes: np.ndarray, bits: int) -> np.ndarray:
    """codes [d_row, d_col] -> qweight int32 [d_col*bits/32, d_row]: column r
    of qweight is row r's codes as an LSB-first stream along the input
    dimension."""
    d_row, d_col = codes.shape
    cols = [_pack_stream(codes[r], bits) for r in range(d_row)]
    return _as_i32([w for c in cols for w in c]).reshape(d_row, -1).T.copy()


def unpack_qweight(qweight: np.ndarray, bits: int, d_col: int) -> np.ndarray:
    qw = np.asarray(qweight).view(np.uint32)
    return np.array([_unpack_stream(qw[:, r], bits, d_col)
                     for r in range(qw.shape[1])], dtype=np.int64)


def pack_qzeros(zeros: np.ndarray, bits: int) -> np.ndarray:
    """zeros [G, d_row] -> qzeros int32 [G, d_row*bits/32], LSB-first along rows."""
    return np.stack([_as_i32(_pack_stream(z, bits)) for z in zeros])


def unpack_qzeros(qzeros: np.ndarray, bits: int, d_row: int) -> np.ndarray:
    qz = np.asarray(qzeros).view(np.uint32)
    return np.array([_unpack_stream(w, bits, d_row) for w in qz], dtype=np.int64)


def packed_bytes(d_row: int, d_col: int, bits: int, group_size: int) -> int:
    """Bytes of qweight + qzeros + scales (fp32) + g_idx for one layer."""
    n_groups = 1 if group_size == -1 else d_col // group_size
    return (d_row * d_col * bits // 8 + n_groups * d_row * bits // 8
            + n_groups * d_row * 4 + d_col * 4)
