"""GPU path vs the CPU oracle at the full sizes of the calibration workloads,
in the configuration the benchmark times (one accumulate over all tokens,
then prepare, quantize and pack through the C ABI).

Every layer shape of the five calibration workloads is covered.  The oracle
cannot redo a whole layer's column loop in seconds, so for each shape it
builds its own fp64 S from all tokens and its own U, compares them with the
GPU's S (whole matrix), order and U, and then solves a seeded sample of rows
exactly (rows are independent): codes, scales, zeros, reconstruction error
and packing of those rows against the GPU's.  Tolerances are those of the
other parity tests (tests/parity.py), with no case held to a lower bar.
"""
import numpy as np
import pytest

import oracle as O
from post_weight_quantization_31_b300 import workloads as wl
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from post_weight_quantization_31_b300 import build_lib
    build_lib.build()


def gpu_layer(inp, exact_diag=None, want_S=False, want_U=False):
    """One solve through the public API; returns host arrays."""
    import torch
    from post_weight_quantization_31_b300 import api
    d_row, d_col = inp.W.shape
    solver = api.LayerSolver(d_row, d_col, inp.cfg, exact_diag=exact_diag)
    solver.reset()
    Xd = torch.from_numpy(inp.X).cuda()
    solver.accumulate(Xd)
    del Xd
    solver.prepare()
    solver.quantize(P.torch_w(inp.W, inp.w_dtype))
    solver.pack()
    solver.check()
    torch.cuda.synchronize()
    o = solver.out
    res = dict(codes=o["codes"].cpu().numpy(), scales=o["scales"].cpu().numpy(),
               zeros=o["zeros"].cpu().numpy().astype(np.int64),
               g_idx=o["g_idx"].cpu().numpy().astype(np.int64),
               perm=solver.perm.cpu().numpy().astype(np.int64),
               qweight=solver.qweight.cpu().numpy(), n=solver.n_seen)
    if want_S:
        res["S"] = solver.S.cpu().numpy()
    if want_U:
        res["U"] = solver.U.cpu().numpy()
    del solver
    torch.cuda.empty_cache()
    return res


def sample_rows(d_row, k, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.sort(rng.choice(d_row, size=k, replace=False))


def check_rows_exact(inp, g, S64, perm, U, rows):
    """Oracle column loop on the sampled rows with the oracle's own U; the
    GPU's codes, scales, zeros and reconstruction error must agree."""
    cfg = inp.cfg
    W = inp.W[rows].astype(np.float64)
    codes_p, scales, zeros, Q_p = O.column_loop(W[:, perm], U, cfg)
    codes = np.empty_like(codes_p)
    codes[:, perm] = codes_p
    Q = np.empty_like(Q_p)
    Q[:, perm] = Q_p
    gc = g["codes"][rows].astype(np.int64)
    same = gc == codes
    assert same.mean() >= P.CODE_MATCH, same.mean()
    assert np.abs(gc - codes).max() <= 1
    gs, gz = g["scales"][:, rows], g["zeros"][:, rows]
    up = P.upstream_groups(gc, codes, perm, cfg.group_size, scales.shape[0])
    srel = np.abs(gs.astype(np.float64) - scales) / np.abs(scales.astype(np.float64))
    assert srel[up].max() <= P.SCALE_RTOL, srel[up].max()
    assert (gz == zeros).mean() >= P.CODE_MATCH
    assert np.abs(gz - zeros).max() <= 1
    eg = P.output_error(inp.W[rows], P.dequantized(gc, gs, gz, g["g_idx"]), S64)
    er = O.recon_error(inp.W[rows], Q, S64)
    assert abs(eg - er) / er <= P.RECON_RTOL, (eg, er)
    # packing of the sampled rows, bit-exact
    assert np.array_equal(P.unpack_columns(g["qweight"][:, rows], cfg.bits, W.shape[1]), gc)


# ------------------------------------------------------------------ all shapes
# (id, inputs, exact fp64 diagonal as the benchmark or API default runs it,
#  sampled rows, key of the calibration set: cases with the same X share the
#  oracle's S and U, which do not depend on bits)
CASES = [
    ("attn_proj_7b", lambda: wl.attn_proj_7b(), False, 48, "attn7b"),
    ("mlp_gate_up_7b", lambda: wl.mlp_7b("gate_up"), None, 32, "mlp_gu"),
    ("mlp_down_7b", lambda: wl.mlp_7b("down"), None, 32, "mlp_down"),
    ("decoder_qkv_7b", lambda: wl.decoder_site_7b("qkv", layer=0), None, 48, "dec_qkv"),
    ("decoder_o_7b", lambda: wl.decoder_site_7b("o", layer=0), None, 48, "dec_o"),
    ("decoder_gate_up_7b", lambda: wl.decoder_site_7b("gate_up", layer=0), None, 32, "dec_gu"),
    ("decoder_down_7b", lambda: wl.decoder_site_7b("down", layer=0), None, 32, "dec_down"),
    ("lowbit_attn_13b_3bit", lambda: wl.lowbit_13b("attn", 3), None, 32, "l13_attn"),
    ("lowbit_attn_13b_2bit", lambda: wl.lowbit_13b("attn", 2), None, 32, "l13_attn"),
    ("lowbit_gate_up_13b_3bit", lambda: wl.lowbit_13b("gate_up", 3), None, 32, "l13_gu"),
    ("lowbit_gate_up_13b_2bit", lambda: wl.lowbit_13b("gate_up", 2), None, 32, "l13_gu"),
    ("lowbit_down_13b_3bit", lambda: wl.lowbit_13b("down", 3), None, 32, "l13_down"),
    ("lowbit_down_13b_2bit", lambda: wl.lowbit_13b("down", 2), None, 32, "l13_down"),
]

_CACHE = {}


def _oracle_factor(key, inp):
    """The oracle's fp64 S from all tokens, its order and its U, shared by
    the cases with the same calibration set."""
    if key not in _CACHE:
        _CACHE.clear()
        S64 = O.hessian_sum_chunked(inp.X)
        perm, _Hp, U = O.prepare(S64, inp.X.shape[1], inp.cfg)
        _CACHE[key] = (S64, perm, U)
    return _CACHE[key]


@pytest.mark.parametrize("name,make,exact_diag,nrows,key", CASES, ids=[c[0] for c in CASES])
def test_full_size_layer_against_oracle(name, make, exact_diag, nrows, key):
    inp = make()
    n = inp.X.shape[1]
    g = gpu_layer(inp, exact_diag=exact_diag, want_S=True, want_U=True)
    S64, perm, U = _oracle_factor(key, inp)
    assert P.s_error(g["S"], S64) < P.s_tol(n)
    assert np.array_equal(g["perm"], perm)
    assert np.array_equal(g["g_idx"], O.group_index(perm, inp.cfg.group_size))
    Ug = g["U"].astype(np.float64)
    assert np.all(np.tril(Ug, -1) == 0) and np.all(np.diag(Ug) > 0)
    assert np.max(np.abs(Ug - U)) / np.max(np.abs(U)) < 2e-4
    assert g["codes"].max() <= (1 << inp.cfg.bits) - 1
    rows = sample_rows(inp.W.shape[0], nrows, seed=17)
    check_rows_exact(inp, g, S64, perm, U, rows)
