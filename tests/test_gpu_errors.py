"""Status codes from the device: non-positive pivots and non-finite inputs
are reported, never trapped, and the context stays usable afterwards."""
import numpy as np
import pytest

from post_weight_quantization_31_b300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from post_weight_quantization_31_b300 import build_lib
    build_lib.build()


def qc(**kw):
    base = dict(bits=4, group_size=128, damp_percent=0.01, blocksize=128, desc_act=False,
                sym=False)
    base.update(kw)
    return wl.QuantConfig(**base)


def test_zero_hessian_is_not_pd_then_damping_fixes_dead_channels():
    import torch
    from post_weight_quantization_31_b300 import api
    d = 256
    S = torch.zeros((d, d), dtype=torch.float32, device="cuda")
    with pytest.raises(api.GPTQError) as e:
        api.prepare_hinv(S, 100, qc())
    assert e.value.code == 2
    # half of the channels dead: singular without damping, fine with it
    X = wl.make_activations(d, 1024, seed=1)
    X[::2] = 0
    S.zero_()
    n = api.hessian_accumulate(torch.from_numpy(X).cuda(), S)
    with pytest.raises(api.GPTQError) as e:
        api.prepare_hinv(S, n, qc(damp_percent=0.0))
    assert e.value.code == 2
    U, perm = api.prepare_hinv(S, n, qc(damp_percent=0.01))
    assert torch.isfinite(U).all()


def test_nonfinite_inputs_are_reported():
    import torch
    from post_weight_quantization_31_b300 import api
    d = 256
    X = wl.make_activations(d, 512, seed=2)
    X[5, 7] = np.inf
    S = torch.zeros((d, d), dtype=torch.float32, device="cuda")
    n = api.hessian_accumulate(torch.from_numpy(X).cuda(), S)
    with pytest.raises(api.GPTQError) as e:
        api.prepare_hinv(S, n, qc())
    assert e.value.code == 3
    X[5, 7] = 1.0
    S.zero_()
    n = api.hessian_accumulate(torch.from_numpy(X).cuda(), S)
    U, perm = api.prepare_hinv(S, n, qc())
    W = torch.zeros((64, d), dtype=torch.float32, device="cuda")
    W[3, 9] = float("nan")
    with pytest.raises(api.GPTQError) as e:
        api.quantize_layer(W, U, perm, qc())
    assert e.value.code == 3
    W[3, 9] = 0.0
    out = api.quantize_layer(W, U, perm, qc())       # context still usable
    assert out["codes"].shape == (64, d)
    api.device_fault()                                # no timeout recorded


def test_status_is_read_later_from_the_workspace():
    """prepare_hinv and quantize_layer return once enqueued; a device-side
    error waits in the call's workspace until workspace_status reads it, and
    it stays with that workspace (another call's workspace reads OK)."""
    import torch
    from post_weight_quantization_31_b300 import api
    d = 256
    S = torch.zeros((d, d), dtype=torch.float32, device="cuda")
    ws_bad = torch.empty(api.prepare_workspace_size(d), dtype=torch.uint8, device="cuda")
    ws_good = torch.empty_like(ws_bad)
    api.prepare_hinv(S, 100, qc(), ws=ws_bad, check=False)          # no exception here
    X = wl.make_activations(d, 1024, seed=3)
    S2 = torch.zeros_like(S)
    n = api.hessian_accumulate(torch.from_numpy(X).cuda(), S2)
    U, perm = api.prepare_hinv(S2, n, qc(), ws=ws_good, check=False)
    with pytest.raises(api.GPTQError) as e:
        api.workspace_status(ws_bad)
    assert e.value.code == 2
    api.workspace_status(ws_good)                                   # OK
    assert torch.isfinite(U).all()


def test_bounded_wait_runs_out_and_is_reported():
    """A bounded wait that runs out is reported as GPTQ_ERR_TIMEOUT and the
    context stays usable.  The dequantization kernel is launched through a
    test hook whose producer issues no copy, with a 1 ms wait limit: the
    compute warps' waits give up with nothing in flight.  The fault word
    reads TIMEOUT once, then OK, and the next normal call is exact."""
    import ctypes

    import torch
    from post_weight_quantization_31_b300 import _lib, api
    from tests import parity as P
    lib = _lib.load()
    f = lib.gptq_internal_dequant_stalled
    f.restype = ctypes.c_int
    vp = ctypes.c_void_p
    f.argtypes = [vp, vp, vp, vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, vp,
                  ctypes.c_uint64, vp]
    d_row, d_col, bits, gs = 64, 512, 4, 128
    rng = np.random.Generator(np.random.PCG64(5))
    codes = rng.integers(0, 16, size=(d_row, d_col)).astype(np.uint8)
    zeros = rng.integers(0, 16, size=(d_col // gs, d_row)).astype(np.uint8)
    scales = rng.uniform(1e-3, 1e-2, size=(d_col // gs, d_row)).astype(np.float32)
    g_idx = (np.arange(d_col) // gs).astype(np.int32)
    qw, qz = api.pack(torch.from_numpy(codes).cuda(), torch.from_numpy(zeros).cuda(), bits, gs)
    sc, gi = torch.from_numpy(scales).cuda(), torch.from_numpy(g_idx).cuda()
    out = torch.zeros((d_row, d_col), dtype=torch.float16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.gptq_device_fault(stream) == 0                       # clean start
    assert f(qw.data_ptr(), qz.data_ptr(), sc.data_ptr(), gi.data_ptr(), d_row, d_col, bits, gs,
             out.data_ptr(), 1_000_000, stream) == 0
    assert lib.gptq_device_fault(stream) == 5                       # GPTQ_ERR_TIMEOUT
    assert lib.gptq_device_fault(stream) == 0                       # read once, then cleared
    W = api.dequantize(qw, qz, sc, gi, d_row, d_col, bits, gs, dtype=torch.float16)
    torch.cuda.synchronize()
    want = P.dequantized(codes, scales, zeros, g_idx).astype(np.float32).astype(np.float16)
    assert np.array_equal(W.cpu().numpy(), want)
    assert lib.gptq_device_fault(stream) == 0
