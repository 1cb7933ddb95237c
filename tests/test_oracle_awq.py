"""Pins of the AWQ oracle (oracle/awq_oracle.py), CPU only: a worked
example derived by hand (tests/golden/awq_salient_example.json), the
reduction to round-to-nearest, the error identity against X itself, the
equivalence of the two scaling directions the pages describe, and
invariances."""
import json
import os

import numpy as np

import oracle as O
from oracle import awq_oracle as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "awq_salient_example.json")


def cfg(**kw):
    return O.OracleConfig(**kw)


def test_hand_worked_example():
    g = json.load(open(GOLDEN))
    W, X = np.array(g["W"]), np.array(g["X"])
    S = X @ X.T
    c = cfg(bits=g["bits"], group_size=g["group_size"], sym=g["sym"])
    res = A.awq_search(W, S, A.channel_rms(X), c)
    assert list(res.salient) == [0]
    for s, e in g["errors_by_s"].items():
        assert abs(res.errors[float(s)] - e) <= 1e-4 * max(e, 1e-3), (s, res.errors[float(s)], e)
    assert res.factor == g["best_s"]
    assert abs(res.error - g["best_error"]) <= 1e-4 * g["best_error"] + 1e-9
    assert abs(res.errors[1.0] - g["rtn_error"]) < 1e-9


def _case(d_row, d_col, n_tok, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    X = rng.standard_normal((d_col, n_tok))
    X[rng.choice(d_col, size=max(1, d_col // 20), replace=False)] *= rng.uniform(10, 50)
    W = rng.standard_normal((d_row, d_col)) * 0.02
    return W, X


def test_factor_one_is_round_to_nearest():
    W, X = _case(16, 256, 512, 1)
    c = cfg(bits=4, group_size=128)
    codes, scales, zeros, W_hat = A.scaled_rtn(W, np.ones(256), c)
    r = O.rtn(W, c)
    assert np.array_equal(codes, r.codes) and np.array_equal(scales, r.scales)
    assert np.array_equal(W_hat, r.Q)


def test_search_never_worse_than_rtn_and_error_identity():
    W, X = _case(24, 256, 1024, 2)
    S = X @ X.T
    c = cfg(bits=3, group_size=64)
    res = A.awq_search(W, S, A.channel_rms(X), c)
    assert res.error <= res.errors[1.0]
    # tr(D S D^T) is the output error measured on X directly
    D = W - res.W_hat
    assert abs(res.error - float(np.sum((D @ X) ** 2))) <= 1e-9 * res.error
    # with outlier channels the search finds a factor that helps
    assert res.factor > 1.0 and res.error < res.errors[1.0]


def test_salient_selection_ties_and_count():
    rms = np.array([1.0, 5.0, 5.0, 0.5, 3.0, 5.0, 0.1, 0.2])
    assert list(A.salient_channels(rms, frac=0.25)) == [1, 2]      # ceil(2): ties -> lower index
    assert list(A.salient_channels(rms, frac=0.05)) == [1]
    assert list(A.salient_channels(rms, frac=0.0)) == []


def test_two_scaling_directions_agree():
    """Salient x 2 (others 1) and others x 1/2 (salient 1) are the same
    relative scaling; powers of two scale exactly, so the codes and the
    effective weights are identical."""
    W, X = _case(16, 256, 256, 3)
    c = cfg(bits=4, group_size=128)
    sal = A.salient_channels(A.channel_rms(X))
    up = np.ones(256)
    up[sal] = 2.0
    down = np.full(256, 0.5)
    down[sal] = 1.0
    a = A.scaled_rtn(W, up, c)
    b = A.scaled_rtn(W, down, c)
    assert np.array_equal(a[0], b[0])
    assert np.array_equal(a[3], b[3])


def test_uniform_statistics_choose_no_scaling_ties():
    """Scaling every channel by the same power of two changes no code: with
    all channels salient the errors tie and the smallest factor is kept."""
    W, X = _case(8, 128, 256, 4)
    S = X @ X.T
    c = cfg(bits=4, group_size=64)
    res = A.awq_search(W, S, np.ones(128), c, frac=1.0, grid=(1.0, 2.0, 4.0))
    assert res.errors[1.0] == res.errors[2.0] == res.errors[4.0]
    assert res.factor == 1.0


def test_rms_statistic_closed_form():
    """RMS = sqrt(mean(x^2)) per channel: [3, -4] -> sqrt(12.5); a channel
    of +-10 (mean 0) is more active than a constant 1."""
    X = np.array([[3.0, -4.0], [10.0, -10.0], [1.0, 1.0]])
    np.testing.assert_allclose(A.channel_rms(X), [np.sqrt(12.5), 10.0, 1.0], rtol=1e-15)
    assert list(A.salient_channels(A.channel_rms(X), frac=0.2)) == [1]


def _awq_pins_fail():
    """Names of the AWQ pins above that fail (run against the current
    oracle functions)."""
    import pytest as _pytest
    failed = []
    for name, fn in [("golden", test_hand_worked_example), ("rtn", test_factor_one_is_round_to_nearest),
                     ("search", test_search_never_worse_than_rtn_and_error_identity),
                     ("ties", test_salient_selection_ties_and_count),
                     ("directions", test_two_scaling_directions_agree),
                     ("uniform", test_uniform_statistics_choose_no_scaling_ties),
                     ("rms", test_rms_statistic_closed_form)]:
        try:
            fn()
        except (AssertionError, Exception):
            failed.append(name)
    return failed


def test_planted_mistakes_fail_a_pin(monkeypatch):
    """Each planted mistake in the AWQ oracle makes at least one pin fail."""
    assert _awq_pins_fail() == []
    real_scaled, real_sal, real_rms = A.scaled_rtn, A.salient_channels, A.channel_rms

    def not_divided_back(W, t, c):          # forgets to divide the effective weights by t
        codes, scales, zeros, W_hat = real_scaled(W, t, c)
        return codes, scales, zeros, W_hat * t[None, :]

    def least_active(rms, frac=0.05):       # picks the quietest channels
        return real_sal(-np.asarray(rms), frac)

    def mean_not_rms(X):                    # signed mean instead of RMS
        return np.abs(np.mean(np.asarray(X, dtype=np.float64), axis=1))

    for name, attr, fake in [("not divided back", "scaled_rtn", not_divided_back),
                             ("least active", "salient_channels", least_active),
                             ("mean not rms", "channel_rms", mean_not_rms)]:
        with monkeypatch.context() as m:
            m.setattr(A, attr, fake)
            assert _awq_pins_fail(), name
    assert (A.scaled_rtn, A.salient_channels, A.channel_rms) == (real_scaled, real_sal, real_rms)
