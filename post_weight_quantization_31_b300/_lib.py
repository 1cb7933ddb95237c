"""ctypes binding of libgptq_b300.so (declarations in include/gptq.h).

Argument marshalling only: every step of the solver runs in the library's
CUDA kernels.  Loading fails loudly when the library has not been built;
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgptq_b300.so")

GPTQ_OK = 0
STATUS_NAMES = {
    0: "GPTQ_OK",
    1: "GPTQ_ERR_INVALID_ARG",
    2: "GPTQ_ERR_NOT_PD",
    3: "GPTQ_ERR_NONFINITE",
    4: "GPTQ_ERR_WORKSPACE",
    5: "GPTQ_ERR_TIMEOUT",
    6: "GPTQ_ERR_CUDA",
    7: "GPTQ_ERR_UNSUPPORTED",
}
W_FP32, W_BF16, W_FP16 = 0, 1, 2
NOALLOC_MAX_D_COL = 1024  # GPTQ_NOALLOC_MAX_D_COL in include/gptq.h

# Every function the header declares, with (restype, argtypes).
_vp, _i64, _i32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t


class GptqConfigC(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("damp_percent", ctypes.c_float), ("blocksize", ctypes.c_int32),
                ("desc_act", ctypes.c_int32), ("sym", ctypes.c_int32)]


_CFGP = ctypes.POINTER(GptqConfigC)

SIGNATURES = {
    "gptq_hessian_accumulate": (_i32, [_vp, _i64, _i64, _i64, _i32, _vp, _vp,
                                       ctypes.POINTER(ctypes.c_int64), _vp]),
    "gptq_prepare_workspace_size": (_sz, [_i64]),
    "gptq_prepare_hinv": (_i32, [_vp, _vp, _i64, _i64, _CFGP, _vp, _vp, _vp, _sz, _vp]),
    "gptq_prepare_hinv_noalloc": (_i32, [_vp, _vp, _i64, _i64, _CFGP, _vp, _vp, _vp]),
    "gptq_quantize_workspace_size": (_sz, [_i64, _i64, _CFGP]),
    "gptq_quantize_layer": (_i32, [_vp, _i32, _i64, _i64, _vp, _vp, _CFGP, _vp, _vp, _vp, _vp,
                                   _vp, _sz, _vp]),
    "gptq_awq_workspace_size": (_sz, [_i64, _i64, _i32]),
    "gptq_awq_search": (_i32, [_vp, _i32, _i64, _i64, _vp, _vp, _CFGP, ctypes.c_float, _vp, _i32, _vp, _vp,
                               _vp, _vp, _vp, _vp, _sz, _vp]),
    "gptq_pack": (_i32, [_vp, _vp, _i64, _i64, _i32, _i32, _vp, _vp, _vp]),
    "gptq_unpack": (_i32, [_vp, _vp, _i64, _i64, _i32, _i32, _vp, _vp, _vp]),
    "gptq_dequantize": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _vp, _vp]),
    "gptq_dequant_matmul": (_i32, [_vp, _i32, _i64, _i64, _vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32,
                                   _vp, _vp]),
    "gptq_status_string": (ctypes.c_char_p, [_i32]),
    "gptq_device_fault": (_i32, [_vp]),
    "gptq_workspace_status": (_i32, [_vp, _vp]),
    "gptq_launch_count": (ctypes.c_uint64, []),
}

_lib = None


def load() -> ctypes.CDLL:
    """Loads the library once; raises if it is missing or incomplete."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is not built: run `python -m post_weight_quantization_31_b300.build_lib`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)  # AttributeError if a declared symbol is missing
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def make_config(cfg) -> GptqConfigC:
    return GptqConfigC(int(cfg.bits), int(cfg.group_size), float(cfg.damp_percent),
                       int(cfg.blocksize), int(bool(cfg.desc_act)), int(bool(cfg.sym)))


def status_name(code: int) -> str:
    return STATUS_NAMES.get(int(code), f"status {code}")
