"""Oracle checks against numbers the pages print (fixtures in tests/golden/)."""
import json
import os

import numpy as np

import oracle as O
import oracle.gptq_oracle as G

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


def test_minmax_worked_example():
    g = load("minmax_rtn_example.json")
    w = np.array([g["values"]], dtype=np.float64)
    bits = g["bits"]
    # The example's grid spans [min, max] only (no zero in range).
    s, z, span = O.quant_params(w, bits, sym=False, include_zero=False)
    levels = O.dequantize_codes(np.arange(1 << bits), s[0], z[0])
    np.testing.assert_allclose(levels, g["printed_levels"],
                               atol=0.5 * 10 ** -g["printed_decimals"])
    q = O.quantize_codes(np.array([g["probe"]]), span, z, bits)
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


def check_grid_examples(quant_params=None, quantize_codes=None):
    """Hand-worked grids (tests/golden/quant_grid_examples.json): the
    symmetric grid at 2, 3 and 4 bits, the asymmetric grid with a range
    that is extended to include zero from either side, and the empty range.
    Returns the names of the cases the oracle gets wrong."""
    quant_params = quant_params or G.quant_params      # looked up at call time
    quantize_codes = quantize_codes or G.quantize_codes
    bad = []
    for c in load("quant_grid_examples.json")["cases"]:
        w = np.array([c["values"]], dtype=np.float64)
        try:
            s, z, span = quant_params(w, c["bits"], c["sym"])
            q = quantize_codes(w, span[:, None], z[:, None], c["bits"])
            lv = O.dequantize_codes(q, s[:, None], z[:, None])[0]
            ok = (np.isclose(float(s[0]), c["scale"], rtol=1e-7, atol=0)
                  and int(z[0]) == c["zero"] and q[0].tolist() == c["codes"]
                  and np.allclose(lv, c["levels"], rtol=1e-7, atol=1e-12))
        except (FloatingPointError, ValueError, ZeroDivisionError):
            ok = False
        if not ok:
            bad.append(c["name"])
    return bad


def test_quantizer_grid_worked_examples():
    assert check_grid_examples() == []
