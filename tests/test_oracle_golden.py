"""Oracle checks against numbers the pages print (fixtures in tests/golden/)."""
import json
import os

import numpy as np

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


def test_minmax_worked_example():
    g = load("minmax_rtn_example.json")
    w = np.array([g["values"]], dtype=np.float64)
    bits = g["bits"]
    # The example's grid spans [min, max] only (no zero in range).
    s, z = O.quant_params(w, bits, sym=False, include_zero=False)
    levels = O.dequantize_codes(np.arange(1 << bits), s[0], z[0])
    np.testing.assert_allclose(levels, g["printed_levels"],
                               atol=0.5 * 10 ** -g["printed_decimals"])
    q = O.quantize_codes(np.array([g["probe"]]), s, z, bits)
    dq = O.dequantize_codes(q, s, z)
    assert np.isclose(dq[0], g["probe_level"])
    assert np.isclose(g["probe"] - dq[0], g["probe_error"])


def test_weight_storage_formula():
    g = load("weight_storage.json")
    n = g["params"]
    for bits, gb in g["gb_per_bits"].items():
        bits = int(bits)
        assert np.isclose(n * bits / 8 / 1e9, gb)
    # Packed 4-bit codes alone are 0.5 byte per weight; scales, zeros and
    # g_idx come on top and shrink as the group grows.
    d_row, d_col = 4096, 4096
    code_bytes = d_row * d_col * 4 // 8
    small, large = g["smaller_group_is_larger"]
    b_small = O.packed_bytes(d_row, d_col, 4, small)
    b_large = O.packed_bytes(d_row, d_col, 4, large)
    assert b_small > b_large > code_bytes
    # 7B at 4-bit g128: 3.5 GB of codes, under 4 GB with group metadata.
    per_weight = b_large / (d_row * d_col)
    assert 3.5 <= n * per_weight / 1e9 <= 4.0
