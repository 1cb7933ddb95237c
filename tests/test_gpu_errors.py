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
