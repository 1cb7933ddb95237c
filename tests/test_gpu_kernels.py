"""Internal kernels checked directly: the 3xTF32 tensor-core GEMM against
an fp64 product."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from post_weight_quantization_31_b300 import _lib, build_lib
    build_lib.build()
    L = _lib.load()
    f = L.gptq_internal_tgemm
    f.restype = ctypes.c_int
    vp, i64, i32, fl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    f.argtypes = [vp, vp, i64, vp, vp, i64, i32, i32, i32, fl, fl, vp, i64, i32, i32, i32, vp]
    return L


def split(x):
    """TF32 hi (10 explicit mantissa bits, ties away from zero) and lo."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    hi = ((u + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32)
    lo = (x.astype(np.float32) - hi).astype(np.float32)
    return hi, lo


@pytest.mark.parametrize("M,N,K,lower,row_off", [(128, 128, 128, 0, 0), (300, 200, 96, 0, 0),
                                                 (1000, 1100, 128, 1, 100), (4096, 3968, 128, 0, 0),
                                                 (256, 640, 40, 1, 384)])
def test_tgemm_3xtf32(lib, M, N, K, lower, row_off):
    import torch
    rng = np.random.Generator(np.random.PCG64(M + N + K))
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((N, K)).astype(np.float32)
    C0 = rng.standard_normal((M, N)).astype(np.float32)
    ld = (K + 3) // 4 * 4
    Ah, Al = split(A)
    Bh, Bl = split(B)

    def dev(x, ldx):
        t = torch.zeros((x.shape[0], ldx), dtype=torch.float32, device="cuda")
        t[:, :x.shape[1]] = torch.from_numpy(x)
        return t
    tAh, tAl, tBh, tBl = dev(Ah, ld), dev(Al, ld), dev(Bh, ld), dev(Bl, ld)
    C = torch.from_numpy(C0).cuda()
    st = lib.gptq_internal_tgemm(tAh.data_ptr(), tAl.data_ptr(), ld, tBh.data_ptr(), tBl.data_ptr(),
                                 ld, M, N, K, -1.0, 1.0, C.data_ptr(), N, lower, row_off, 0,
                                 torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    got = C.cpu().numpy().astype(np.float64)
    want = C0.astype(np.float64) - A.astype(np.float64) @ B.astype(np.float64).T
    if lower:
        rows = np.arange(M)[:, None] + row_off
        cols = np.arange(N)[None, :]
        want = np.where(cols <= rows, want, C0)
    scale = np.abs(A).astype(np.float64) @ np.abs(B).astype(np.float64).T + np.abs(C0)
    err = np.max(np.abs(got - want) / scale)
    assert err < 2e-6, err
