"""AWQ scale search on the GPU against the CPU oracle (oracle/awq_oracle.py)
on the same seeded inputs: the salient channels, every candidate's layer
output error, the chosen factor, and the codes, scales and zero points of
W diag(t).

Tolerances: errors within 1e-4 relative (the GPU's S is the tensor-core fp32
sum, within ~1e-5 of the exact one, and the error products run in 3xTF32);
the chosen factor is the oracle's, unless the two candidates' oracle errors
are within that tolerance of each other; codes, zeros and scales at the
bar of the GPTQ parity tests (round-to-nearest has no cascades, so codes
must in fact match except at fp32 near-ties)."""
import numpy as np
import pytest

import oracle as O
from oracle import awq_oracle as A
from post_weight_quantization_31_b300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu

ERR_RTOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from post_weight_quantization_31_b300 import build_lib
    build_lib.build()


def qc(**kw):
    base = dict(bits=4, group_size=128, damp_percent=0.01, blocksize=128, desc_act=False, sym=False)
    base.update(kw)
    return wl.QuantConfig(**base)


def run(W, w_dtype, X, cfg, frac=0.05):
    import torch
    from post_weight_quantization_31_b300 import api
    d_col = X.shape[0]
    S = torch.zeros((d_col, d_col), dtype=torch.float32, device="cuda")
    diag = torch.zeros(d_col, dtype=torch.float64, device="cuda")
    api.hessian_accumulate(torch.from_numpy(X).cuda(), S, diag)
    out = api.awq_search(P.torch_w(W, w_dtype), S, diag, cfg, salient_frac=frac)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in out.items()}
    S64 = O.hessian_sum(X)
    ref = A.awq_search(W, S64, A.channel_rms(X), cfg, frac=frac)
    return g, ref, S64


def check(g, ref, W, S64, cfg):
    grid = np.array(A.SCALE_GRID)
    want = np.array([ref.errors[float(s)] for s in grid])
    np.testing.assert_allclose(g["errors"], want, rtol=ERR_RTOL)
    s_gpu = float(g["t"].max())
    if s_gpu != ref.factor:
        # a near tie: the GPU's choice must be as good as the oracle's
        assert abs(ref.errors[s_gpu] - ref.error) <= ERR_RTOL * ref.error, (s_gpu, ref.factor)
        return
    # the salient set and the factor (t = s on the salient channels)
    if ref.factor != 1.0:
        assert np.array_equal(np.flatnonzero(g["t"] != 1.0), ref.salient)
    np.testing.assert_array_equal(g["t"], ref.t.astype(np.float32))
    codes = g["codes"].astype(np.int64)
    assert (codes == ref.codes).mean() >= P.CODE_MATCH
    assert np.abs(codes - ref.codes).max() <= 1
    assert (g["zeros"].astype(np.int64) == ref.zeros).mean() >= P.CODE_MATCH
    srel = np.abs(g["scales"].astype(np.float64) - ref.scales) / ref.scales
    assert srel.max() <= P.SCALE_RTOL
    # the GPU's effective weights reach the oracle's error
    gi = (np.arange(W.shape[1]) // (W.shape[1] if cfg.group_size == -1 else cfg.group_size))
    W_hat = P.dequantized(codes, g["scales"], g["zeros"], gi) / g["t"].astype(np.float64)[None, :]
    eg = P.output_error(W, W_hat, S64)
    assert abs(eg - ref.error) <= 1e-3 * ref.error


CASES = [
    # (name, W, w_dtype, X, cfg)
    ("tiny_outliers", lambda: wl.tiny_layer().W, "fp32", lambda: wl.tiny_layer().X, dict()),
    ("sym_g64_bf16", lambda: wl.make_weight(128, 1024, seed=91, dtype="bf16"), "bf16",
     lambda: wl.make_activations(1024, 4096, seed=92, outlier_frac=0.02, outlier_scale=(10.0, 50.0)),
     dict(sym=True, group_size=64)),
    ("per_row_3bit", lambda: wl.make_weight(64, 512, seed=93, dtype="bf16"), "bf16",
     lambda: wl.make_activations(512, 2048, seed=94, n_outliers=6, outlier_scale=30.0),
     dict(bits=3, group_size=-1)),
    ("student_t_2bit_g32", lambda: wl.make_weight(96, 768, seed=95, dtype="bf16"), "bf16",
     lambda: wl.make_activations(768, 3000, seed=96, kind="student_t"),
     dict(bits=2, group_size=32, sym=True)),
]


@pytest.mark.parametrize("name,mkW,w_dtype,mkX,kw", CASES, ids=[c[0] for c in CASES])
def test_awq_search_matches_oracle(name, mkW, w_dtype, mkX, kw):
    W, X, cfg = mkW(), mkX(), qc(**kw)
    g, ref, S64 = run(W, w_dtype, X, cfg)
    check(g, ref, W, S64, cfg)


def test_awq_picks_scaling_when_outliers_dominate():
    """With a few channels scaled x20 the best factor is above 1, and the
    AWQ error is below plain round-to-nearest (the pages' reason for AWQ)."""
    inp = wl.tiny_layer()
    g, ref, S64 = run(inp.W, "fp32", inp.X, qc())
    assert ref.factor > 1.0
    assert float(g["t"].max()) > 1.0
    assert g["errors"].min() < g["errors"][0]          # candidate 0 is s = 1 (plain RTN)


def test_awq_full_salient_set_of_one_channel():
    """frac small enough that one channel is salient (ceil rounds up)."""
    W = wl.make_weight(64, 256, seed=97, dtype="bf16")
    X = wl.make_activations(256, 1024, seed=98, n_outliers=1, outlier_scale=40.0)
    cfg = qc(group_size=64)
    g, ref, S64 = run(W, "bf16", X, cfg, frac=1e-3)
    assert len(ref.salient) == 1
    check(g, ref, W, S64, cfg)
