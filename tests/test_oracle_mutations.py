"""Planted mistakes in the oracle must each fail at least one pin.

Each mutation patches one step of the oracle (on the CPU) and re-runs the
relevant pin checks; a pin set that passes a broken oracle would not pin it.
"""
import numpy as np
import pytest

import oracle as O
import oracle.gptq_oracle as G
from post_weight_quantization_31_b300 import workloads as wl
from tests.test_oracle_golden import check_grid_examples
from tests.test_oracle_pins import _ls_check


def cfg(**kw):
    base = dict(bits=4, group_size=32, damp_percent=0.01, blocksize=128,
                desc_act=True, sym=False)
    base.update(kw)
    return O.OracleConfig(**base)


def pins_hold():
    """A compact run of P1, P2, P3, P4, I1, the nearest-level pin and the
    hand-worked quantizer grids; returns the names of the pins that fail."""
    failed = ["grid: " + name for name in check_grid_examples()]
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
    s, z, span = G.quant_params(w, 4, False)
    q = G.quantize_codes(w, span[:, None], z[:, None], 4)
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
                       lambda w, span, z, bits: np.clip(np.floor(
                           ((1 << bits) - 1) * (np.asarray(w, np.float64) / span)
                       ).astype(np.int64) + z, 0, (1 << bits) - 1)),
    "hinv_not_factored": ("hinv_upper", lambda H: np.triu(np.linalg.inv(H))),
}


def _mutant_quant_params(mistake: str):
    """The quantizer grid with one planted mistake (R6-R8 otherwise)."""
    def quant_params(w, bits, sym, include_zero=True):
        maxq = (1 << bits) - 1
        w64 = np.asarray(w, dtype=np.float64)
        xmin, xmax = w64.min(axis=1), w64.max(axis=1)
        if include_zero and mistake != "zero_clamp_dropped":
            xmin, xmax = np.minimum(xmin, 0.0), np.maximum(xmax, 0.0)
        with np.errstate(all="ignore"):
            if sym:
                a = np.maximum(np.abs(xmin), np.abs(xmax))
                if mistake != "empty_range_kept":
                    a = np.where(a == 0, 1.0, a)
                span = a if mistake == "sym_scale_a_over_maxq" else 2.0 * a
                zero = np.full(w64.shape[0], maxq // 2 if mistake == "sym_zero_maxq_half"
                               else (maxq + 1) // 2, dtype=np.int64)
            else:
                if mistake != "empty_range_kept":
                    deg = xmin == xmax
                    xmin, xmax = np.where(deg, -1.0, xmin), np.where(deg, 1.0, xmax)
                span = xmax - xmin
                zero = np.nan_to_num(np.rint(maxq * (-xmin / span))).astype(np.int64)
            return (span / maxq).astype(np.float32), zero, span
    return quant_params


def _mutant_codes(w, span, z, bits):
    with np.errstate(all="ignore"):
        t = np.nan_to_num(np.rint(((1 << bits) - 1) * (np.asarray(w, np.float64) / span)))
    return np.clip(t.astype(np.int64) + z, 0, (1 << bits) - 1)


def test_grid_mutant_without_a_mistake_passes(monkeypatch):
    """Control: the mutant grid with no mistake planted passes every pin, so
    a failure below comes from the planted mistake alone."""
    monkeypatch.setattr(G, "quant_params", _mutant_quant_params("none"))
    monkeypatch.setattr(G, "quantize_codes", _mutant_codes)
    assert pins_hold() == []


GRID_MUTATIONS = ("sym_scale_a_over_maxq", "sym_zero_maxq_half", "zero_clamp_dropped",
                  "empty_range_kept")


@pytest.mark.parametrize("name", sorted(MUTATIONS) + list(GRID_MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    if name in GRID_MUTATIONS:
        monkeypatch.setattr(G, "quant_params", _mutant_quant_params(name))
        monkeypatch.setattr(G, "quantize_codes", _mutant_codes)
    else:
        attr, fn = MUTATIONS[name]
        monkeypatch.setattr(G, attr, fn)
    failed = pins_hold()
    assert failed != [], name
    if name in GRID_MUTATIONS:
        # the hand-worked grids are the pins that catch a wrong grid
        assert any(f.startswith("grid: ") for f in failed), (name, failed)
