"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, independent of the oracle's own code paths.

P1  H = I reduces GPTQ to round-to-nearest exactly.
P2  on tiny layers the compensation after every quantized column equals the
    least-squares optimum of the remaining weights, solved directly.
P3  lazy-batched and unbatched column loops agree to fp64 round-off.
P4  GPTQ's reconstruction error is below RTN's on seeded cases.
I1  invariance to the scale of S.   I2  two-column closed form.
I3  row independence.               I4  U^T U H = I, both U routes agree.
I7  brute force over all code vectors on tiny rows.
"""
import itertools

import numpy as np
import pytest

import oracle as O
from post_weight_quantization_31_b300 import workloads as wl


def cfg(**kw):
    base = dict(bits=4, group_size=128, damp_percent=0.01, blocksize=128,
                desc_act=False, sym=False)
    base.update(kw)
    return O.OracleConfig(**base)


def spd_from_x(X):
    return O.hessian_sum(X), X.shape[1]


# ------------------------------------------------------------------ P1
@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("gs", [32, 128, -1])
@pytest.mark.parametrize("desc_act", [False, True])
def test_p1_identity_hessian_is_rtn(bits, sym, gs, desc_act):
    d_row, d_col = 48, 256
    W = wl.make_weight(d_row, d_col, seed=11 + bits, dtype="bf16")
    n = 1000
    S = np.eye(d_col) * (n / 2.0)          # H = (2/n) S = I
    c = cfg(bits=bits, sym=sym, group_size=gs, desc_act=desc_act)
    g = O.quantize_layer(W, S, n, c)
    r = O.rtn(W, c)
    assert np.array_equal(g.perm, np.arange(d_col))   # all diagonals tie
    assert np.array_equal(g.codes, r.codes)
    assert np.array_equal(g.scales, r.scales)
    assert np.array_equal(g.zeros, r.zeros)
    assert np.array_equal(g.Q, r.Q)


# ------------------------------------------------------------------ P2
def _ls_check(W0p, Hp, c, rtol=1e-10):
    """After each quantized column, the remaining weights must equal the
    direct least-squares optimum: argmin_wF (w - w0)^T H (w - w0) with the
    quantized columns held at their dequantized values."""
    d_col = W0p.shape[1]
    U = O.hinv_upper(Hp)
    states = {}

    def trace(j, W):
        states[j] = W.copy()

    codes, scales, zeros, Q = O.column_loop(W0p, U, c, blocksize=1, trace=trace)
    worst = 0.0
    for j in range(d_col - 1):
        Qs, F = np.arange(j + 1), np.arange(j + 1, d_col)
        delta_Q = Q[:, Qs] - W0p[:, Qs]
        # H_FF (w_F - w0_F) + H_FQ (w_Q - w0_Q) = 0
        rhs = -(Hp[np.ix_(F, Qs)] @ delta_Q.T)
        wF = W0p[:, F] + np.linalg.solve(Hp[np.ix_(F, F)], rhs).T
        got = states[j][:, F]
        err = np.max(np.abs(got - wF)) / max(np.max(np.abs(wF)), 1e-300)
        worst = max(worst, err)
    return worst <= rtol, worst


@pytest.mark.parametrize("d_col", [2, 3, 5, 8])
@pytest.mark.parametrize("gs", [-1, 2])
def test_p2_compensation_is_least_squares(d_col, gs):
    if gs != -1 and d_col % gs:
        pytest.skip("group must divide d_col")
    X = wl.make_correlated_activations(d_col, 64, seed=100 + d_col)
    S, n = spd_from_x(X)
    c = cfg(bits=3, group_size=gs, damp_percent=0.05, blocksize=1)
    H = O.damped_hessian(S, n, c.damp_percent)
    W0 = wl.make_weight(6, d_col, seed=7, dtype="fp32").astype(np.float64)
    ok, worst = _ls_check(W0, H, c)
    assert ok, worst


# ------------------------------------------------------------------ P3
@pytest.mark.parametrize("gs", [32, 128, -1])
@pytest.mark.parametrize("desc_act", [False, True])
def test_p3_lazy_batch_equals_unbatched(gs, desc_act):
    d_row, d_col = 24, 256
    X = wl.make_correlated_activations(d_col, 512, seed=5)
    S, n = spd_from_x(X)
    W = wl.make_weight(d_row, d_col, seed=6, dtype="bf16")
    c = cfg(group_size=gs, desc_act=desc_act)
    outs = [O.quantize_layer(W, S, n, c, blocksize=b) for b in (1, 8, 128, d_col)]
    for o in outs[1:]:
        assert np.array_equal(o.codes, outs[0].codes)
        assert np.array_equal(o.scales, outs[0].scales)
        np.testing.assert_allclose(o.Q, outs[0].Q, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------ P4
CASES_P4 = [
    ("iid_outliers", lambda: wl.make_activations(256, 2048, 21, n_outliers=4,
                                                 outlier_scale=20.0)),
    ("correlated", lambda: wl.make_correlated_activations(256, 1024, 22)),
    ("lowrank", lambda: wl.make_lowrank_activations(256, 1024, 23)),
    ("student_t", lambda: wl.make_activations(256, 2048, 24, kind="student_t")),
]


@pytest.mark.parametrize("name,mk", CASES_P4, ids=[c[0] for c in CASES_P4])
@pytest.mark.parametrize("bits,sym,gs,desc_act", [(4, False, 128, False),
                                                  (4, True, 128, False),
                                                  (3, True, 64, True),
                                                  (2, True, 64, True),
                                                  (4, False, -1, True)])
def test_p4_gptq_error_below_rtn(name, mk, bits, sym, gs, desc_act):
    X = mk()
    S, n = spd_from_x(X)
    W = wl.make_weight(64, X.shape[0], seed=25, dtype="bf16")
    c = cfg(bits=bits, sym=sym, group_size=gs, desc_act=desc_act)
    g = O.quantize_layer(W, S, n, c)
    r = O.rtn(W, c)
    eg, er = O.recon_error(W, g.Q, S), O.recon_error(W, r.Q, S)
    assert eg <= er, (eg, er)


def test_p4_tiny_workload():
    inp = wl.tiny_layer()
    S, n = spd_from_x(inp.X)
    g = O.quantize_layer(inp.W, S, n, inp.cfg)
    r = O.rtn(inp.W, inp.cfg)
    assert O.recon_error(inp.W, g.Q, S) < O.recon_error(inp.W, r.Q, S)


# ------------------------------------------------------------------ I1
def test_i1_scale_invariance():
    X = wl.make_correlated_activations(128, 512, seed=31)
    S, n = spd_from_x(X)
    W = wl.make_weight(16, 128, seed=32, dtype="bf16")
    c = cfg(group_size=32, desc_act=True)
    a = O.quantize_layer(W, S, n, c)
    b = O.quantize_layer(W, 37.5 * S, n, c)
    d = O.quantize_layer(W, S, 3 * n, c)
    for o in (b, d):
        assert np.array_equal(o.codes, a.codes)
        assert np.array_equal(o.perm, a.perm)
        np.testing.assert_allclose(o.Q, a.Q, rtol=1e-12)


# ------------------------------------------------------------------ I2
def test_i2_two_column_closed_form():
    rng = np.random.Generator(np.random.PCG64(41))
    for _ in range(20):
        A = rng.standard_normal((2, 2))
        H = A @ A.T + 0.1 * np.eye(2)
        w = rng.standard_normal((5, 2)) * 0.02
        c = cfg(bits=3, group_size=-1, blocksize=1)
        U = O.hinv_upper(H)
        codes, scales, zeros, Q = O.column_loop(w, U, c, blocksize=1)
        s, z, span = O.quant_params(w, 3, False)
        q0 = O.quantize_codes(w[:, 0], span, z, 3)
        dq0 = s.astype(np.float64) * (q0 - z)
        w1 = w[:, 1] + (w[:, 0] - dq0) * H[0, 1] / H[1, 1]
        assert np.array_equal(codes[:, 0], q0)
        assert np.array_equal(codes[:, 1], O.quantize_codes(w1, span, z, 3))


# ------------------------------------------------------------------ I3
def test_i3_row_independence():
    X = wl.make_correlated_activations(256, 512, seed=51)
    S, n = spd_from_x(X)
    W = wl.make_weight(40, 256, seed=52, dtype="bf16")
    c = cfg(group_size=64, desc_act=True)
    full = O.quantize_layer(W, S, n, c)
    rows = np.array([3, 17, 18, 39, 0])
    sub = O.quantize_layer(W, S, n, c, rows=rows)
    assert np.array_equal(sub.codes, full.codes[rows])
    assert np.array_equal(sub.scales, full.scales[:, rows])
    np.testing.assert_array_equal(sub.Q, full.Q[rows])


# ------------------------------------------------------------------ I4
@pytest.mark.parametrize("n", [1, 2, 7, 40])
def test_i4_inverse_cholesky_factor(n):
    X = wl.make_correlated_activations(n, 4 * n + 8, seed=60 + n)
    S, m = spd_from_x(X)
    H = O.damped_hessian(S, m, 0.01)
    U = O.hinv_upper(H)
    assert np.allclose(np.tril(U, -1), 0.0)
    assert np.all(np.diag(U) > 0)
    np.testing.assert_allclose(U.T @ U @ H, np.eye(n), atol=1e-10)
    np.testing.assert_allclose(O.hinv_upper_reverse(H), U, rtol=1e-9, atol=1e-12)


def test_i4_not_positive_definite_raises():
    H = np.diag([1.0, -1.0, 2.0])
    with pytest.raises(np.linalg.LinAlgError):
        O.hinv_upper(H)
    with pytest.raises(np.linalg.LinAlgError):
        O.hinv_upper_reverse(H)


# ------------------------------------------------------------------ I7
@pytest.mark.parametrize("d_col", [1, 2, 3, 4])
def test_i7_bruteforce_lower_bound(d_col):
    X = wl.make_correlated_activations(d_col, 32, seed=70 + d_col)
    S, n = spd_from_x(X)
    c = cfg(bits=2, group_size=-1, damp_percent=0.0, blocksize=1)
    W = wl.make_weight(1, d_col, seed=71, dtype="fp32")
    g = O.quantize_layer(W, S, n, c)
    s, z = g.scales[0], g.zeros[0]
    best = np.inf
    for qv in itertools.product(range(4), repeat=d_col):
        Qv = s.astype(np.float64)[:, None] * (np.array(qv)[None, :] - z[:, None])
        best = min(best, O.recon_error(W, Qv, S))
    eg = O.recon_error(W, g.Q, S)
    assert best <= eg * (1 + 1e-12)
    if d_col == 1:      # a single weight: rounding to nearest is optimal
        assert np.isclose(best, eg, rtol=1e-12)


# ------------------------------------------------------------------ a2 pieces
def test_damping_and_order():
    S = np.diag([4.0, 1.0, 4.0, 9.0, 1.0])
    n = 8                      # H = S/4 -> diag [1, .25, 1, 2.25, .25], mean 0.95
    H = O.damped_hessian(S, n, 0.1)
    np.testing.assert_allclose(np.diag(H), [1.095, 0.345, 1.095, 2.345, 0.345])
    perm = O.act_order(H, True)
    assert perm.tolist() == [3, 0, 2, 1, 4]        # stable on ties
    assert O.act_order(H, False).tolist() == [0, 1, 2, 3, 4]


def test_group_index_maps_original_columns():
    perm = np.array([3, 0, 2, 1])
    assert O.group_index(perm, 2).tolist() == [0, 1, 1, 0]
    assert O.group_index(perm, -1).tolist() == [0, 0, 0, 0]


def test_hessian_entry_matches_sum():
    X = wl.make_activations(16, 100, seed=81)
    S = O.hessian_sum(X)
    assert S[3, 7] == O.hessian_entry(X, 3, 7)
    Xf = X.astype(np.float64)
    assert S[5, 5] == sum(float(v) * float(v) for v in Xf[5])


def test_chunked_hessian_helpers_match_brute_force():
    """The chunked fp64 sums used at full size against explicit Python loops."""
    X = wl.make_activations(12, 50, seed=82, n_outliers=2, outlier_scale=20.0)
    Xf = [[float(v) for v in row] for row in X]
    brute = np.array([[sum(a * b for a, b in zip(Xf[i], Xf[j])) for j in range(12)]
                      for i in range(12)])
    np.testing.assert_allclose(O.hessian_sum_chunked(X, chunk=7), brute, rtol=1e-12, atol=0)
    np.testing.assert_allclose(O.hessian_diag(X, chunk=9), np.diag(brute), rtol=1e-12, atol=0)
    np.testing.assert_allclose(O.hessian_columns(X, [3, 0, 11], chunk=13), brute[:, [3, 0, 11]],
                               rtol=1e-12, atol=0)


def test_act_order_from_diagonal():
    d = np.array([1.0, 3.0, 3.0, 0.5, 2.0])
    assert list(O.act_order_diag(d, True)) == [1, 2, 4, 0, 3]   # tie keeps 1 before 2
    assert list(O.act_order_diag(d, False)) == [0, 1, 2, 3, 4]
    assert list(O.act_order(np.diag(d), True)) == [1, 2, 4, 0, 3]
