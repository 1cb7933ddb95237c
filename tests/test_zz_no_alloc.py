"""gptq_prepare_hinv_noalloc: the prepare step for callers that cannot
allocate device memory (code inside another framework's memory pool, or a
latency-critical path where cudaMalloc/cudaFree would synchronize the
device).  Its scratch space is a fixed array inside the library, so its
results must equal those of gptq_prepare_hinv with a caller workspace, call
after call, whatever the previous call left in that array.

This file is collected last on purpose: if it fails, every other test has
already run."""
import ctypes

import numpy as np
import pytest

import oracle as O
from post_weight_quantization_31_b300 import _lib
from post_weight_quantization_31_b300 import workloads as wl


def qc(**kw):
    base = dict(bits=4, group_size=128, damp_percent=0.01, blocksize=128, desc_act=False,
                sym=False)
    base.update(kw)
    return wl.QuantConfig(**base)


def test_noalloc_rejects_d_col_beyond_its_scratch():
    """Host-side check, before anything touches the (fake) pointers."""
    from post_weight_quantization_31_b300 import build_lib
    build_lib.build()
    lib = _lib.load()
    c = _lib.make_config(qc())
    fake = 1 << 20
    d = _lib.NOALLOC_MAX_D_COL + 32
    st = lib.gptq_prepare_hinv_noalloc(fake, None, d, 1000, ctypes.byref(c), fake, fake, None)
    assert st == 4  # GPTQ_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_matches_workspace_version_two_calls_in_a_row():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from post_weight_quantization_31_b300 import api, build_lib
    build_lib.build()
    lib = _lib.load()
    stream = torch.cuda.current_stream().cuda_stream
    # Two calls in a row on the shared scratch: the larger one first, so that
    # the second runs on what the first left behind.
    for d_col, kw in ((1024, dict(desc_act=True)), (544, dict(group_size=32))):
        cfg = qc(**kw)
        X = wl.make_activations(d_col, 4 * d_col, seed=d_col + 11, outlier_frac=0.01)
        S = torch.zeros((d_col, d_col), dtype=torch.float32, device="cuda")
        diag = torch.zeros(d_col, dtype=torch.float64, device="cuda")
        n = api.hessian_accumulate(torch.from_numpy(X).cuda(), S, diag)
        U_ref, perm_ref = api.prepare_hinv(S, n, cfg, diag=diag)
        U = torch.full((d_col, d_col), float("nan"), dtype=torch.float32, device="cuda")
        perm = torch.full((d_col,), -1, dtype=torch.int32, device="cuda")
        c = _lib.make_config(cfg)
        st = lib.gptq_prepare_hinv_noalloc(S.data_ptr(), diag.data_ptr(), d_col, n,
                                           ctypes.byref(c), U.data_ptr(), perm.data_ptr(),
                                           stream)
        assert st == 0, _lib.status_name(st)
        torch.cuda.synchronize()
        # The prepare step has no floating-point atomics: with the same inputs
        # it is deterministic, so the fixed scratch array must give exactly the
        # caller-workspace result, whatever the previous call left in it.
        assert np.array_equal(perm.cpu().numpy(), perm_ref.cpu().numpy())
        Ug, Ur = U.cpu().numpy(), U_ref.cpu().numpy()
        assert np.array_equal(Ug.view(np.uint32), Ur.view(np.uint32)), d_col
        # and both agree with the oracle's factor of the same Hessian
        perm_o, Hp, U_o = O.prepare(O.hessian_sum(X), n, cfg)
        assert np.array_equal(perm.cpu().numpy(), perm_o)
        err = np.max(np.abs(Ug.astype(np.float64) - U_o)) / np.max(np.abs(U_o))
        assert err < 2e-4, (d_col, err)
