"""Python API over the C ABI: the same four calls, taking torch tensors.

PyTorch only provides device memory and the current CUDA stream; every step
of the solver runs in libgptq_b300.so.  All tensors must live on the current
CUDA device.
"""
from __future__ import annotations

import ctypes
import dataclasses

import torch

from . import _lib
from .workloads import QuantConfig


class GPTQError(RuntimeError):
    def __init__(self, code: int, where: str):
        lib = _lib.load()
        msg = lib.gptq_status_string(int(code)).decode()
        super().__init__(f"{where}: {_lib.status_name(code)} ({msg})")
        self.code = int(code)


def _check(code: int, where: str) -> None:
    if int(code) != _lib.GPTQ_OK:
        raise GPTQError(code, where)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _need(t: torch.Tensor, dtype, name: str, shape=None) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _contig(t: torch.Tensor, name: str) -> None:
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def n_groups(group_size: int, d_col: int) -> int:
    return 1 if group_size == -1 else d_col // group_size


def launch_count() -> int:
    return int(_lib.load().gptq_launch_count())


# ----------------------------------------------------------------------- a1
def hessian_accumulate(X: torch.Tensor, S: torch.Tensor, diag: torch.Tensor | None = None,
                       token_major: bool = False) -> int:
    """S += X X^T (and diag += sum_t X^2 in fp64 if given).  X: fp16
    [d_col, n_tok] with unit stride along tokens, or with token_major=True
    [n_tok, d_col] with unit stride along channels (a [tokens, features]
    activation tensor).  Returns n_tok."""
    lib = _lib.load()
    _need(X, torch.float16, "X")
    if X.dim() != 2 or X.stride(1) != 1:
        raise ValueError("X must be 2-D with a unit inner stride")
    n_tok, d_col = X.shape if token_major else X.shape[::-1]
    if X.stride(0) % 8 != 0 or X.data_ptr() % 16 != 0:
        # The library reads X with TMA, which needs 16-byte aligned rows:
        # copy into storage whose row stride is a multiple of 8 halves.
        rows, cols = X.shape
        ld = (cols + 7) // 8 * 8
        Xp = torch.empty((rows, ld), dtype=X.dtype, device=X.device)
        Xp[:, :cols].copy_(X)
        X = Xp[:, :cols]
    _need(S, torch.float32, "S", (d_col, d_col))
    _contig(S, "S")
    if diag is not None:
        _need(diag, torch.float64, "diag", (d_col,))
    n = ctypes.c_int64(0)
    _check(lib.gptq_hessian_accumulate(X.data_ptr(), d_col, n_tok, X.stride(0), int(token_major),
                                       S.data_ptr(), _ptr(diag), ctypes.byref(n), _stream()),
           "gptq_hessian_accumulate")
    return int(n.value)


# ----------------------------------------------------------------------- a2
def prepare_workspace_size(d_col: int) -> int:
    return int(_lib.load().gptq_prepare_workspace_size(d_col))


def workspace_status(ws: torch.Tensor, where: str = "gptq_workspace_status") -> None:
    """Waits for the current stream and raises GPTQError if the last
    prepare/quantize call on `ws` reported an error on the device."""
    _check(_lib.load().gptq_workspace_status(ws.data_ptr(), _stream()), where)


def prepare_hinv(S: torch.Tensor, n_seen: int, cfg: QuantConfig, diag: torch.Tensor | None = None,
                 U: torch.Tensor | None = None, perm: torch.Tensor | None = None,
                 ws: torch.Tensor | None = None, check: bool = True):
    """Returns (U, perm): U fp32 [d, d] upper with H_perm^-1 = U^T U.

    The library call is asynchronous; with check=True (the default) this
    waits for it and raises on a device-side error (NOT_PD, NONFINITE,
    TIMEOUT).  With check=False the caller reads the status later with
    workspace_status(ws)."""
    lib = _lib.load()
    d = S.shape[0]
    _need(S, torch.float32, "S", (d, d))
    dev = S.device
    U = torch.empty((d, d), dtype=torch.float32, device=dev) if U is None else U
    perm = torch.empty(d, dtype=torch.int32, device=dev) if perm is None else perm
    need = prepare_workspace_size(d)
    ws = torch.empty(need, dtype=torch.uint8, device=dev) if ws is None else ws
    c = _lib.make_config(cfg)
    _check(lib.gptq_prepare_hinv(S.data_ptr(), _ptr(diag), d, int(n_seen), ctypes.byref(c),
                                 U.data_ptr(), perm.data_ptr(), ws.data_ptr(), ws.numel(),
                                 _stream()), "gptq_prepare_hinv")
    if check:
        workspace_status(ws, "gptq_prepare_hinv")
    return U, perm


def prepare_hinv_noalloc(S: torch.Tensor, n_seen: int, cfg: QuantConfig, U: torch.Tensor,
                         perm: torch.Tensor, diag: torch.Tensor | None = None):
    """prepare_hinv for callers that cannot allocate device memory: U and perm
    are the caller's, the scratch space is the library's own fixed array
    (d_col <= 1024).  Calls whose GPU work overlaps share that array and race."""
    lib = _lib.load()
    d = S.shape[0]
    _need(S, torch.float32, "S", (d, d))
    _need(U, torch.float32, "U", (d, d))
    _need(perm, torch.int32, "perm", (d,))
    c = _lib.make_config(cfg)
    _check(lib.gptq_prepare_hinv_noalloc(S.data_ptr(), _ptr(diag), d, int(n_seen), ctypes.byref(c),
                                         U.data_ptr(), perm.data_ptr(), _stream()),
           "gptq_prepare_hinv_noalloc")
    return U, perm


# ----------------------------------------------------------------------- a3/a4
def quantize_workspace_size(d_row: int, d_col: int, cfg: QuantConfig) -> int:
    c = _lib.make_config(cfg)
    return int(_lib.load().gptq_quantize_workspace_size(d_row, d_col, ctypes.byref(c)))


_WDT = {torch.float32: _lib.W_FP32, torch.bfloat16: _lib.W_BF16, torch.float16: _lib.W_FP16}


def quantize_layer(W: torch.Tensor, U: torch.Tensor, perm: torch.Tensor, cfg: QuantConfig,
                   out: dict | None = None, ws: torch.Tensor | None = None,
                   check: bool = True) -> dict:
    """Returns dict(codes uint8 [d_row, d_col] original order, scales fp32
    [G, d_row], zeros uint8 [G, d_row], g_idx int32 [d_col]).  `check` as
    for prepare_hinv."""
    lib = _lib.load()
    if W.dtype not in _WDT:
        raise ValueError("W must be fp32, bf16 or fp16")
    _contig(W, "W")
    d_row, d_col = W.shape
    _need(U, torch.float32, "U", (d_col, d_col))
    _contig(U, "U")
    _need(perm, torch.int32, "perm", (d_col,))
    dev = W.device
    G = n_groups(cfg.group_size, d_col)
    out = {} if out is None else out
    codes = out.setdefault("codes", torch.empty((d_row, d_col), dtype=torch.uint8, device=dev))
    scales = out.setdefault("scales", torch.empty((G, d_row), dtype=torch.float32, device=dev))
    zeros = out.setdefault("zeros", torch.empty((G, d_row), dtype=torch.uint8, device=dev))
    g_idx = out.setdefault("g_idx", torch.empty(d_col, dtype=torch.int32, device=dev))
    need = quantize_workspace_size(d_row, d_col, cfg)
    ws = torch.empty(need, dtype=torch.uint8, device=dev) if ws is None else ws
    c = _lib.make_config(cfg)
    _check(lib.gptq_quantize_layer(W.data_ptr(), _WDT[W.dtype], d_row, d_col, U.data_ptr(),
                                   perm.data_ptr(), ctypes.byref(c), codes.data_ptr(),
                                   scales.data_ptr(), zeros.data_ptr(), g_idx.data_ptr(),
                                   ws.data_ptr(), ws.numel(), _stream()), "gptq_quantize_layer")
    if check:
        workspace_status(ws, "gptq_quantize_layer")
    return out


# ----------------------------------------------------------------------- AWQ
AWQ_GRID = tuple(1.0 + 0.25 * i for i in range(13))      # 1, 1.25, ..., 4


def awq_search(W: torch.Tensor, S: torch.Tensor, diag: torch.Tensor, cfg: QuantConfig,
               salient_frac: float = 0.05, grid=AWQ_GRID, ws: torch.Tensor | None = None,
               check: bool = True) -> dict:
    """AWQ scale search (see gptq_awq_search in include/gptq.h).  Returns
    dict(codes uint8 [d_row, d_col] of W diag(t), scales fp32 [G, d_row],
    zeros uint8 [G, d_row], t fp32 [d_col], errors fp64 [n_grid])."""
    lib = _lib.load()
    if W.dtype not in _WDT:
        raise ValueError("W must be fp32, bf16 or fp16")
    _contig(W, "W")
    d_row, d_col = W.shape
    _need(S, torch.float32, "S", (d_col, d_col))
    _contig(S, "S")
    _need(diag, torch.float64, "diag", (d_col,))
    dev = W.device
    G = n_groups(cfg.group_size, d_col)
    g = (ctypes.c_float * len(grid))(*[float(v) for v in grid])
    out = {"codes": torch.empty((d_row, d_col), dtype=torch.uint8, device=dev),
           "scales": torch.empty((G, d_row), dtype=torch.float32, device=dev),
           "zeros": torch.empty((G, d_row), dtype=torch.uint8, device=dev),
           "t": torch.empty(d_col, dtype=torch.float32, device=dev),
           "errors": torch.empty(len(grid), dtype=torch.float64, device=dev)}
    need = int(lib.gptq_awq_workspace_size(d_row, d_col, len(grid)))
    ws = torch.empty(need, dtype=torch.uint8, device=dev) if ws is None else ws
    c = _lib.make_config(cfg)
    _check(lib.gptq_awq_search(W.data_ptr(), _WDT[W.dtype], d_row, d_col, S.data_ptr(), diag.data_ptr(),
                               ctypes.byref(c), float(salient_frac), ctypes.cast(g, ctypes.c_void_p),
                               len(grid), out["codes"].data_ptr(), out["scales"].data_ptr(),
                               out["zeros"].data_ptr(), out["t"].data_ptr(), out["errors"].data_ptr(),
                               ws.data_ptr(), ws.numel(), _stream()), "gptq_awq_search")
    if check:
        workspace_status(ws, "gptq_awq_search")
    return out


# ----------------------------------------------------------------------- a5
def pack(codes: torch.Tensor, zeros: torch.Tensor, bits: int, group_size: int,
         qweight: torch.Tensor | None = None, qzeros: torch.Tensor | None = None):
    lib = _lib.load()
    d_row, d_col = codes.shape
    G = n_groups(group_size, d_col)
    dev = codes.device
    qweight = (torch.empty((d_col * bits // 32, d_row), dtype=torch.int32, device=dev)
               if qweight is None else qweight)
    qzeros = (torch.empty((G, d_row * bits // 32), dtype=torch.int32, device=dev)
              if qzeros is None else qzeros)
    _check(lib.gptq_pack(codes.data_ptr(), zeros.data_ptr(), d_row, d_col, bits, group_size,
                         qweight.data_ptr(), qzeros.data_ptr(), _stream()), "gptq_pack")
    return qweight, qzeros


def unpack(qweight: torch.Tensor, qzeros: torch.Tensor, d_row: int, d_col: int, bits: int,
           group_size: int):
    lib = _lib.load()
    G = n_groups(group_size, d_col)
    dev = qweight.device
    codes = torch.empty((d_row, d_col), dtype=torch.uint8, device=dev)
    zeros = torch.empty((G, d_row), dtype=torch.uint8, device=dev)
    _check(lib.gptq_unpack(qweight.data_ptr(), qzeros.data_ptr(), d_row, d_col, bits, group_size,
                           codes.data_ptr(), zeros.data_ptr(), _stream()), "gptq_unpack")
    return codes, zeros


_OUT_DT = {torch.float32: _lib.W_FP32, torch.bfloat16: _lib.W_BF16, torch.float16: _lib.W_FP16}


def dequantize(qweight: torch.Tensor, qzeros: torch.Tensor, scales: torch.Tensor,
               g_idx: torch.Tensor, d_row: int, d_col: int, bits: int, group_size: int,
               dtype=torch.float16, out: torch.Tensor | None = None) -> torch.Tensor:
    """Dense weights [d_row, d_col] (original column order) from the packed layer."""
    lib = _lib.load()
    if dtype not in _OUT_DT:
        raise ValueError("dtype must be fp32, bf16 or fp16")
    out = torch.empty((d_row, d_col), dtype=dtype, device=qweight.device) if out is None else out
    _check(lib.gptq_dequantize(qweight.data_ptr(), qzeros.data_ptr(), scales.data_ptr(),
                               g_idx.data_ptr(), d_row, d_col, bits, group_size, _OUT_DT[dtype],
                               out.data_ptr(), _stream()), "gptq_dequantize")
    return out


def dequant_matmul(X: torch.Tensor, qweight: torch.Tensor, qzeros: torch.Tensor, scales: torch.Tensor,
                   g_idx: torch.Tensor, d_row: int, d_col: int, bits: int, group_size: int,
                   out: torch.Tensor | None = None) -> torch.Tensor:
    """Y [M, d_row] fp32 = X [M, d_col] (fp16 or bf16) times the packed
    layer's dequantized weights, transposed."""
    lib = _lib.load()
    if X.dtype not in (torch.float16, torch.bfloat16) or X.dim() != 2 or X.stride(1) != 1:
        raise ValueError("X must be a 2-D fp16/bf16 tensor with unit column stride")
    M = X.shape[0]
    out = torch.empty((M, d_row), dtype=torch.float32, device=X.device) if out is None else out
    _check(lib.gptq_dequant_matmul(X.data_ptr(), _OUT_DT[X.dtype], M, X.stride(0), qweight.data_ptr(),
                                   qzeros.data_ptr(), scales.data_ptr(), g_idx.data_ptr(), d_row, d_col,
                                   bits, group_size, out.data_ptr(), _stream()), "gptq_dequant_matmul")
    return out


def device_fault() -> None:
    _check(_lib.load().gptq_device_fault(_stream()), "gptq_device_fault")


# ----------------------------------------------------------------------- whole layer
@dataclasses.dataclass
class LayerResult:
    qweight: torch.Tensor
    qzeros: torch.Tensor
    scales: torch.Tensor
    g_idx: torch.Tensor
    codes: torch.Tensor
    zeros: torch.Tensor
    perm: torch.Tensor
    U: torch.Tensor


class LayerSolver:
    """Owns the device buffers for one layer shape and runs the four calls.

    Buffers are allocated once (through PyTorch) and reused, so repeated
    solves allocate nothing.
    """

    def __init__(self, d_row: int, d_col: int, cfg: QuantConfig, device="cuda",
                 exact_diag: bool | None = None):
        self.d_row, self.d_col, self.cfg = d_row, d_col, cfg
        self.device = torch.device(device)
        dev = self.device
        self.exact_diag = bool(cfg.desc_act) if exact_diag is None else exact_diag
        G = n_groups(cfg.group_size, d_col)
        self.S = torch.zeros((d_col, d_col), dtype=torch.float32, device=dev)
        self.diag = (torch.zeros(d_col, dtype=torch.float64, device=dev)
                     if self.exact_diag else None)
        self.n_seen = 0
        self.U = torch.empty((d_col, d_col), dtype=torch.float32, device=dev)
        self.perm = torch.empty(d_col, dtype=torch.int32, device=dev)
        self.ws_prep = torch.empty(prepare_workspace_size(d_col), dtype=torch.uint8, device=dev)
        self.ws_quant = torch.empty(quantize_workspace_size(d_row, d_col, cfg), dtype=torch.uint8,
                                    device=dev)
        self.out = {
            "codes": torch.empty((d_row, d_col), dtype=torch.uint8, device=dev),
            "scales": torch.empty((G, d_row), dtype=torch.float32, device=dev),
            "zeros": torch.empty((G, d_row), dtype=torch.uint8, device=dev),
            "g_idx": torch.empty(d_col, dtype=torch.int32, device=dev),
        }
        self.qweight = torch.empty((d_col * cfg.bits // 32, d_row), dtype=torch.int32, device=dev)
        self.qzeros = torch.empty((G, d_row * cfg.bits // 32), dtype=torch.int32, device=dev)

    def staging(self, tokens: int, count: int = 2) -> list:
        """`count` device buffers [d_col, tokens] fp16 for chunked host input."""
        cur = getattr(self, "_stage", None)
        if cur is None or cur[0].shape[1] < tokens or len(cur) != count:
            self._stage = [torch.empty((self.d_col, tokens), dtype=torch.float16,
                                       device=self.device) for _ in range(count)]
        return self._stage

    def w_buffer(self, dtype) -> torch.Tensor:
        cur = getattr(self, "_wbuf", None)
        if cur is None or cur.dtype != dtype:
            self._wbuf = torch.empty((self.d_row, self.d_col), dtype=dtype, device=self.device)
        return self._wbuf

    def reset(self) -> None:
        self.S.zero_()
        if self.diag is not None:
            self.diag.zero_()
        self.n_seen = 0

    def accumulate(self, X: torch.Tensor) -> None:
        self.n_seen += hessian_accumulate(X, self.S, self.diag)

    def prepare(self) -> None:
        """Enqueues the prepare call (asynchronous; see check())."""
        prepare_hinv(self.S, self.n_seen, self.cfg, diag=self.diag, U=self.U, perm=self.perm,
                     ws=self.ws_prep, check=False)

    def quantize(self, W: torch.Tensor) -> None:
        """Enqueues the quantize call (asynchronous; see check())."""
        quantize_layer(W, self.U, self.perm, self.cfg, out=self.out, ws=self.ws_quant, check=False)

    def check(self) -> None:
        """Waits for the current stream and raises GPTQError if the last
        prepare or quantize reported an error on the device."""
        workspace_status(self.ws_prep, "gptq_prepare_hinv")
        workspace_status(self.ws_quant, "gptq_quantize_layer")

    def pack(self) -> None:
        pack(self.out["codes"], self.out["zeros"], self.cfg.bits, self.cfg.group_size,
             qweight=self.qweight, qzeros=self.qzeros)

    def solve(self, W: torch.Tensor, X: torch.Tensor | None = None) -> LayerResult:
        """Accumulate X (if given), then prepare, quantize and pack."""
        if X is not None:
            self.accumulate(X)
        self.prepare()
        self.quantize(W)
        self.pack()
        self.check()
        return self.result()

    def result(self) -> LayerResult:
        return LayerResult(qweight=self.qweight, qzeros=self.qzeros, scales=self.out["scales"],
                           g_idx=self.out["g_idx"], codes=self.out["codes"],
                           zeros=self.out["zeros"], perm=self.perm, U=self.U)


def quantize_layer_from_host(W_host: torch.Tensor, X_chunks, cfg: QuantConfig,
                             solver: LayerSolver | None = None, copy_streams: int = 2) -> dict:
    """End to end from host memory.

    X_chunks: sequence of host fp16 tensors [d_col, t_i] (contiguous; pinned
    for asynchronous copies), e.g. one per batch of calibration sequences.
    Chunks are copied to the device on `copy_streams` side streams (chunk i
    on stream i mod copy_streams, so that several copy engines can run at
    once) into rotating staging buffers, overlapped with the Hessian
    accumulation of the chunks already copied; then the layer is solved and
    the packed result (qweight, qzeros, scales, g_idx) is returned in host
    memory.
    """
    d_row, d_col = W_host.shape
    solver = solver or LayerSolver(d_row, d_col, cfg)
    solver.reset()
    dev = solver.device
    compute = torch.cuda.current_stream(dev)
    n_copy = max(1, int(copy_streams))
    copies = getattr(solver, "_copy_streams", None)
    if copies is None or len(copies) != n_copy:
        copies = [torch.cuda.Stream(dev) for _ in range(n_copy)]
        solver._copy_streams = copies
    cap = max(int(c.shape[1]) for c in X_chunks)
    cap = (cap + 7) // 8 * 8
    # One staging buffer more than there are copy streams lets each copy
    # stream start its next chunk while the Hessian of its last one runs.
    stage = solver.staging(cap, count=n_copy + 2)
    ready = [torch.cuda.Event() for _ in stage]
    free = [torch.cuda.Event() for _ in stage]
    used = [False] * len(stage)
    W_dev = solver.w_buffer(W_host.dtype)
    for ci, chunk in enumerate(X_chunks):
        if chunk.shape[0] != d_col or chunk.dtype != torch.float16:
            raise ValueError("each X chunk must be fp16 [d_col, t]")
        b = ci % len(stage)
        cs = copies[ci % n_copy]
        t = int(chunk.shape[1])
        buf = stage[b][:, :t]
        with torch.cuda.stream(cs):
            if used[b]:
                cs.wait_event(free[b])
            buf.copy_(chunk, non_blocking=True)
            ready[b].record(cs)
        used[b] = True
        compute.wait_event(ready[b])
        solver.accumulate(buf)
        free[b].record(compute)
    # W is needed only by the quantize step: its copy goes last, beside the
    # Hessian of the last chunk and the prepare step.
    wcs = copies[len(X_chunks) % n_copy]
    with torch.cuda.stream(wcs):
        W_dev.copy_(W_host, non_blocking=True)
    w_ready = torch.cuda.Event()
    w_ready.record(wcs)
    compute.wait_event(w_ready)
    solver.prepare()
    solver.quantize(W_dev)
    solver.pack()
    r = solver.result()
    # The packed result goes to fresh pinned host tensors on the compute
    # stream, behind the solve; check() then waits for that stream once and
    # raises if the device reported an error.
    out = {}
    for name, t in (("qweight", r.qweight), ("qzeros", r.qzeros), ("scales", r.scales),
                    ("g_idx", r.g_idx)):
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t, non_blocking=True)
        out[name] = h
    solver.check()
    return out
