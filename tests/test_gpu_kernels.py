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
                                                 (256, 640, 40, 1, 384),
                                                 # CTA pairs sharing B: an odd number of tile rows
                                                 # (the last pair half beyond M), ragged N and K
                                                 (1100, 2500, 96, 0, 0), (4096, 1536, 512, 0, 0)])
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


@pytest.mark.parametrize("M,N,K,lower,row_off,pri_nt,max_ctas", [
    (3968, 4096, 128, 1, 128, 1, 147),    # prepare step 0 at d = 4096
    (1920, 4096, 128, 1, 2176, 17, 0),    # a middle step
    (256, 4096, 128, 1, 3840, 30, 5),     # the last step with a rest subset
    (700, 900, 64, 0, 0, 3, 0),           # ragged, no triangle
    (128, 512, 96, 1, 384, 3, 0)])        # one tile row: the rest is empty
def test_tgemm_tile_subsets_partition_the_update(lib, M, N, K, lower, row_off, pri_nt, max_ctas):
    """The prepare's update GEMM runs as two launches over complementary tile
    subsets (the next step's row and column blocks first, then the rest, the
    latter on fewer CTAs).  Together they must give exactly the single
    launch's result, every tile once: the same tile arithmetic, bit for bit."""
    import torch
    f = lib.gptq_internal_tgemm_subset
    f.restype = ctypes.c_int
    vp, i64, i32, fl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    f.argtypes = [vp, vp, i64, vp, vp, i64, i32, i32, i32, fl, fl, vp, i64, i32, i32, i32, i32, i32, i32,
                  vp, vp]
    rng = np.random.Generator(np.random.PCG64(M * 7 + N + K))
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((N, K)).astype(np.float32)
    C0 = rng.standard_normal((M, N)).astype(np.float32)
    Ah, Al = split(A)
    Bh, Bl = split(B)
    tAh, tAl, tBh, tBl = (torch.from_numpy(x).cuda() for x in (Ah, Al, Bh, Bl))
    st = torch.cuda.current_stream().cuda_stream
    out = {}
    counts = {}
    for subsets in ((0,), (1, 2), (2, 1)):
        C = torch.from_numpy(C0).cuda()
        for sub in subsets:
            n = ctypes.c_int(-1)
            rc = f(tAh.data_ptr(), tAl.data_ptr(), K, tBh.data_ptr(), tBl.data_ptr(), K, M, N, K, -1.0, 1.0,
                   C.data_ptr(), N, lower, row_off, 0, sub, pri_nt, max_ctas if sub == 2 else 0,
                   ctypes.byref(n), st)
            assert rc == 0
            counts[sub] = n.value
        torch.cuda.synchronize()
        out[subsets] = C.cpu().numpy()
    assert counts[1] + counts[2] == counts[0]
    assert counts[1] > 0
    assert np.array_equal(out[(1, 2)], out[(0,)])
    assert np.array_equal(out[(2, 1)], out[(0,)])
    # and the single launch is the update itself
    want = C0.astype(np.float64) - A.astype(np.float64) @ B.astype(np.float64).T
    if lower:
        want = np.where(np.arange(N)[None, :] <= np.arange(M)[:, None] + row_off, want, C0)
    scale = np.abs(A).astype(np.float64) @ np.abs(B).astype(np.float64).T + np.abs(C0)
    assert np.max(np.abs(out[(0,)] - want) / scale) < 2e-6


def test_grid_quotient_equals_ieee_division(lib):
    """The column loop decides codes on maxq * (w / span) with w / span taken
    from the reciprocal plus one exact-residual correction; it must equal
    CUDA's IEEE division bit for bit, on random operands and on the exact
    midpoints of the symmetric grid (w = -span/2)."""
    import torch
    f = lib.gptq_internal_div_span
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p]
    rng = np.random.Generator(np.random.PCG64(99))
    n = 1 << 20
    span = rng.uniform(1e-4, 0.5, n).astype(np.float32)
    x = (rng.standard_normal(n) * 0.05).astype(np.float32)
    k = n // 8
    x[:k] = -0.5 * span[:k]                        # exact midpoints
    x[k:2 * k] = span[k:2 * k]                     # quotient exactly 1
    span[2 * k:3 * k] = np.float32(2.0) ** rng.integers(-12, 0, k).astype(np.float32)
    tx, ts = torch.from_numpy(x).cuda(), torch.from_numpy(span).cuda()
    qg, qi = torch.empty_like(tx), torch.empty_like(tx)
    assert f(tx.data_ptr(), ts.data_ptr(), n, qg.data_ptr(), qi.data_ptr(),
             torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    a, b = qg.cpu().numpy(), qi.cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert np.all(a[:k] == -0.5) and np.all(a[k:2 * k] == 1.0)
    # and IEEE division itself: the fp64 quotient rounded once to fp32
    want = (x.astype(np.float64) / span.astype(np.float64)).astype(np.float32)
    assert np.array_equal(b, want)
