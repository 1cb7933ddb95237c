"""I6: packing is a bijection, with hand-checkable word layouts."""
import itertools

import numpy as np
import pytest

import oracle as O


def u32(a):
    return np.asarray(a).view(np.uint32)


def test_4bit_lsb_first_word():
    codes = np.array([[1, 2, 3, 4, 5, 6, 7, 8]])
    qw = O.pack_qweight(codes, 4)
    assert qw.shape == (1, 1)
    assert u32(qw)[0, 0] == 0x87654321


def test_2bit_and_8bit_words():
    c2 = np.array([[3] + [0] * 14 + [1]])
    assert u32(O.pack_qweight(c2, 2))[0, 0] == 0x40000003
    c8 = np.array([[0x11, 0x22, 0x33, 0xFF]])
    assert u32(O.pack_qweight(c8, 8))[0, 0] == 0xFF332211


def test_3bit_stream_across_words():
    ones = np.full((1, 32), 7)
    assert u32(O.pack_qweight(ones, 3))[:, 0].tolist() == [0xFFFFFFFF] * 3
    c = np.zeros((1, 32), dtype=np.int64)
    c[0, 10] = 7           # bits 30..32: straddles word 0 and word 1
    assert u32(O.pack_qweight(c, 3))[:, 0].tolist() == [0xC0000000, 0x1, 0x0]
    c = np.zeros((1, 32), dtype=np.int64)
    c[0, 21] = 5           # bits 63..65: 1 in word 1 bit 31, 0b10 in word 2
    assert u32(O.pack_qweight(c, 3))[:, 0].tolist() == [0x0, 0x80000000, 0x2]
    c = np.zeros((1, 32), dtype=np.int64)
    c[0, 31] = 6           # bits 93..95
    assert u32(O.pack_qweight(c, 3))[:, 0].tolist() == [0, 0, 0xC0000000]


def test_3bit_against_bigint_stream():
    rng = np.random.Generator(np.random.PCG64(3))
    c = rng.integers(0, 8, size=(5, 64))
    qw = u32(O.pack_qweight(c, 3))
    for r in range(5):
        big = sum(int(v) << (3 * k) for k, v in enumerate(c[r]))
        words = [(big >> (32 * i)) & 0xFFFFFFFF for i in range(6)]
        assert qw[:, r].tolist() == words


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_roundtrip_exhaustive(bits):
    vals = np.arange(1 << bits)
    per = 32  # a multiple of 32/bits words for every width
    rows = []
    for v, pos in itertools.product(vals, range(per)):
        r = np.zeros(per, dtype=np.int64)
        r[pos] = v
        rows.append(r)
    codes = np.array(rows)
    qw = O.pack_qweight(codes, bits)
    assert qw.shape == (per * bits // 32, codes.shape[0])
    assert np.array_equal(O.unpack_qweight(qw, bits, per), codes)
    zeros = codes[:, :].T.copy()           # [G=32, d_row]
    qz = O.pack_qzeros(zeros[:, :((codes.shape[0] // 32) * 32)], bits)
    back = O.unpack_qzeros(qz, bits, (codes.shape[0] // 32) * 32)
    assert np.array_equal(back, zeros[:, :back.shape[1]])


def test_rejects_out_of_range_code():
    with pytest.raises(ValueError):
        O.pack_qweight(np.array([[16] + [0] * 7]), 4)


def test_dequantize_worked_example():
    """Two rows, four columns, two groups scattered by g_idx (act-order):
    W[r, c] = s[g, r] * (q[r, c] - z[g, r]) with g = g_idx[c], by hand."""
    codes = np.array([[3, 0, 15, 8], [1, 2, 7, 9]])
    scales = np.array([[0.5, 0.25], [2.0, 0.125]])      # [G=2, d_row=2]
    zeros = np.array([[8, 4], [7, 1]])
    g_idx = np.array([1, 0, 0, 1])
    want = np.array([[2.0 * (3 - 7), 0.5 * (0 - 8), 0.5 * (15 - 8), 2.0 * (8 - 7)],
                     [0.125 * (1 - 1), 0.25 * (2 - 4), 0.25 * (7 - 4), 0.125 * (9 - 1)]])
    np.testing.assert_array_equal(O.dequantize(codes, scales, zeros, g_idx), want)
    for dt in ("fp32", "fp16", "bf16"):
        np.testing.assert_array_equal(O.dequantize_as(codes, scales, zeros, g_idx, dt), want)


def test_bf16_rounding_ties_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to the even mantissa (1.0);
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: ties to 1 + 2^-6.
    x = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -20, -(1 + 2.0 ** -8)],
                 dtype=np.float32)
    np.testing.assert_array_equal(O.round_bf16(x), np.array([1.0, 1 + 2.0 ** -6, 1 + 2.0 ** -7, -1.0],
                                                            dtype=np.float32))


def test_dequant_matmul_brute_force():
    """Y[m][n] = sum_k X[m][k] * W[n][k] with W[n][k] = s[g_k][n] * (q[n][k] - z[g_k][n])
    stored in fp32, by loops."""
    rng = np.random.Generator(np.random.PCG64(4))
    M, N, K, bits = 3, 4, 6, 3
    codes = rng.integers(0, 1 << bits, size=(N, K))
    zeros = rng.integers(0, 1 << bits, size=(2, N))
    scales = rng.uniform(0.1, 1.0, size=(2, N)).astype(np.float32)
    g_idx = np.array([1, 0, 1, 1, 0, 0])
    X = rng.standard_normal((M, K)).astype(np.float16).astype(np.float64)
    want = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            for k in range(K):
                g = g_idx[k]
                w = np.float32(scales[g, n]) * np.float32(codes[n, k] - zeros[g, n])  # W stored in fp32
                want[m, n] += X[m, k] * float(w)
    got = O.dequant_matmul(X, codes, scales, zeros, g_idx, "fp32")
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
