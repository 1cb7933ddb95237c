"""The NumPy helpers that measure GPU outputs (tests/parity.py) agree with
the oracle on oracle-made data, so GPU outputs never need to pass through
the oracle."""
import numpy as np
import pytest

import oracle as O
from tests import parity as P


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_unpack_helpers_invert_the_oracle_packers(bits):
    rng = np.random.Generator(np.random.PCG64(bits))
    codes = rng.integers(0, 1 << bits, size=(64, 160))
    zeros = rng.integers(0, 1 << bits, size=(5, 64))
    assert np.array_equal(P.unpack_columns(O.pack_qweight(codes, bits), bits, 160), codes)
    assert np.array_equal(P.unpack_rows(O.pack_qzeros(zeros, bits), bits, 64), zeros)


def test_dequantized_and_output_error_match_the_oracle():
    rng = np.random.Generator(np.random.PCG64(1))
    codes = rng.integers(0, 16, size=(8, 64))
    zeros = rng.integers(0, 16, size=(4, 8))
    scales = rng.uniform(0.01, 0.1, size=(4, 8)).astype(np.float32)
    g_idx = O.group_index(rng.permutation(64), 16)
    Q = P.dequantized(codes, scales, zeros, g_idx)
    assert np.array_equal(Q, O.dequantize(codes, scales, zeros, g_idx))
    X = rng.standard_normal((64, 100))
    W = rng.standard_normal((8, 64)) * 0.1
    S = X @ X.T
    assert abs(P.output_error(W, Q, S) - O.recon_error(W, Q, S)) <= 1e-12 * O.recon_error(W, Q, S)
    assert abs(P.output_error(W, Q, S) - float(np.sum(((W - Q) @ X) ** 2))) <= 1e-9 * P.output_error(W, Q, S)
