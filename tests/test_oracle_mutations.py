"""Planted mistakes in the oracle must each fail at least one pin.

Each mutation patches one step of the oracle (on the CPU) and re-runs the
relevant pin checks; a pin set that passes a broken oracle would not pin it.
"""
import numpy as np
import pytest

import oracle as O
import oracle.gptq_oracle as G
from post_weight_quantization_31_b300 import workloads as wl
from tests.test_oracle_pins import _ls_check


def cfg(**kw):
    base = dict(bits=4, group_size=32, damp_percent=0.01, blocksize=128,
                desc_act=True, sym=False)
    base.update(kw)
    return O.OracleConfig(**base)


def pins_hold():
    """A compact run of P1, P2, P3, P4, I1, I2 and the nearest-level pin;
    returns the names of the pins that fail."""
    failed = []
    # P1
    W = wl.make_weight(8, 64, seed=1, dtype="bf16")
    c = cfg()
    g = G.quantize_layer(W, np.eye(64) * 50.0, 100, c)
    r = G.rtn(W, c)
    if not (np.array_equal(g.codes, r.codes) and np.array_equal(g.Q, r.Q)):
        failed.append("P1")
    # P2
    X = wl.make_correlated_activations(6, 40, seed=2)
    S, n = G.hessian_sum(X), X.shape[1]
    H = G.damped_hessian(S, n, 0.05)
    W0 = wl.make_weight(4, 6, seed=3, dtype="fp32").astype(np.float64)
    try:
        ok, _ = _ls_check(W0, H, cfg(bits=3, group_size=-1, blocksize=1))
    except Exception:
        ok = False
    if not ok:
        failed.append("P2")
    # P3 / P4 / I1
    X = wl.make_correlated_activations(128, 512, seed=4)
    S, n = G.hessian_sum(X), X.shape[1]
    W = wl.make_weight(16, 128, seed=5, dtype="bf16")
    a = G.quantize_layer(W, S, n, c, blocksize=1)
    b = G.quantize_layer(W, S, n, c, blocksize=128)
    if not (np.array_equal(a.codes, b.codes) and np.allclose(a.Q, b.Q, rtol=1e-12)):
        failed.append("P3")
    if not G.recon_error(W, b.Q, S) <= G.recon_error(W, G.rtn(W, c).Q, S):
        failed.append("P4")
    d = G.quantize_layer(W, S, 3 * n, c)
    if not np.array_equal(d.codes, b.codes):
        failed.append("I1")
    # nearest level: every in-range weight lands on its nearest grid point
    rng = np.random.Generator(np.random.PCG64(6))
    w = rng.standard_normal((50, 16))
    s, z = G.quant_params(w, 4, False)
    q = G.quantize_codes(w, s[:, None], z[:, None], 4)
    dq = G.dequantize_codes(q, s[:, None], z[:, None])
    grid = s[:, None, None].astype(np.float64) * (np.arange(16)[None, None, :] - z[:, None, None])
    nearest = np.min(np.abs(w[:, :, None] - grid), axis=2)
    if not np.allclose(np.abs(w - dq), nearest, rtol=0, atol=1e-7 * np.abs(w).max()):
        failed.append("nearest")
    return failed


def test_unmodified_oracle_passes():
    assert pins_hold() == []


MUTATIONS = {
    "update_sign": ("obq_update",
                    lambda W, e, U, j, k1, k2: W.__setitem__(
                        (slice(None), slice(k1, k2)),
                        W[:, k1:k2] + np.outer(e, U[j, k1:k2]))),
    "update_transposed": ("obq_update",
                          lambda W, e, U, j, k1, k2: W.__setitem__(
                              (slice(None), slice(k1, k2)),
                              W[:, k1:k2] - np.outer(e, U[k1:k2, j]))),
    "drop_trailing": ("lazy_trailing_update", lambda W, Err, U, i1, i2: None),
    "error_not_scaled": ("obq_error", lambda w, dq, u: w - dq),
    "damp_from_S": ("damped_hessian",
                    lambda S, n, d: (2.0 / n) * S + d * np.mean(np.diag(S)) * np.eye(S.shape[0])),
    "floor_rounding": ("quantize_codes",
                       lambda w, s, z, bits: np.clip(np.floor(
                           (np.asarray(w, np.float64).astype(np.float32)
                            * (np.float32(1) / np.asarray(s, np.float32))).astype(np.float32)
                       ).astype(np.int64) + z, 0, (1 << bits) - 1)),
    "hinv_not_factored": ("hinv_upper", lambda H: np.triu(np.linalg.inv(H))),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(G, attr, fn)
    assert pins_hold() != [], name
