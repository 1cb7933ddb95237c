"""The prepare's trailing update runs, at every 128-column step, as two
launches of the update GEMM over complementary tile subsets: first the tiles
the next step reads (its block row and its block column), then the rest,
beside the next step's factor kernel.  Each launch picks its tile width
(128 x 128, or 128 x 64 when it would fill fewer than half the SMs) on its
own, so the two may use different widths.  These tests check, on the host
and for every step of several sizes, that the two launches together update
every entry of the lower triangle exactly once, that the first holds all
the next step reads, and that the single launch they replace covers the
same entries.  No GPU: the library's planner is called, nothing launches."""
import ctypes

import numpy as np
import pytest

from post_weight_quantization_31_b300 import _lib

NB = 128
SMS = 148


@pytest.fixture(scope="module")
def lib():
    from post_weight_quantization_31_b300 import build_lib
    build_lib.build()
    lib = _lib.load()
    f = lib.gptq_internal_tgemm_tiles
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 8 + [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    return lib


def plan(lib, M, N, lower, row_off, subset, pri_nt, sms=SMS):
    bn = ctypes.c_int(0)
    n = lib.gptq_internal_tgemm_tiles(M, N, lower, row_off, 0, subset, pri_nt, sms, ctypes.byref(bn),
                                      None, 0)
    assert n >= 0
    coords = np.zeros(2 * max(n, 1), np.int32)
    n2 = lib.gptq_internal_tgemm_tiles(M, N, lower, row_off, 0, subset, pri_nt, sms, ctypes.byref(bn),
                                       coords.ctypes.data, n)
    assert n2 == n
    return bn.value, coords[: 2 * n].reshape(n, 2)


def chunk_counts(bn, tiles, m_tiles, n_chunks):
    """How often each 128-row x 64-column chunk is covered by the tiles."""
    cnt = np.zeros((m_tiles, n_chunks), np.int32)
    w = bn // 64
    for mt, nt in tiles:
        assert 0 <= mt < m_tiles and 0 <= nt * w < n_chunks
        cnt[mt, nt * w: nt * w + w] += 1
    return cnt


def lower_chunks(M, N, row_off):
    """Chunks holding an entry (row_off + r, c) with c <= row_off + r."""
    m_tiles, n_chunks = (M + 127) // 128, (N + 63) // 64
    mt = np.arange(m_tiles)[:, None]
    q = np.arange(n_chunks)[None, :]
    last_row = np.minimum(row_off + 128 * mt + 127, row_off + M - 1)
    return (64 * q <= last_row) & (64 * q < N)


def prepare_steps(d):
    for k in range(0, d, NB):
        b = min(NB, d - k)
        M = d - k - b
        if M > 0:
            yield k, b, M


@pytest.mark.parametrize("d", [160, 544, 1056, 4096, 5120, 11008])
def test_update_subsets_partition_the_lower_triangle(lib, d):
    for k, b, M in prepare_steps(d):
        row_off, pri_nt = k + b, (k + b) // NB
        m_tiles, n_chunks = (M + 127) // 128, (d + 63) // 64
        want = lower_chunks(M, d, row_off)
        cover = {}
        for sub in (0, 1, 2):
            bn, tiles = plan(lib, M, d, 1, row_off, sub, pri_nt)
            assert bn in (64, 128)
            # no tile twice within a launch
            assert len({(int(a), int(c)) for a, c in tiles}) == len(tiles)
            cover[sub] = chunk_counts(bn, tiles, m_tiles, n_chunks)
        both = cover[1] + cover[2]
        ctx = (d, k)
        # every chunk of the lower triangle exactly once, by the pair and by
        # the single launch; nothing above it twice
        assert np.all(both[want] == 1), ctx
        assert np.all(cover[0][want] == 1), ctx
        assert np.all(both <= 1) and np.all(cover[0] <= 1), ctx
        # a tile lies wholly above the diagonal only where a 128-wide tile's
        # second half does (at most one 64-column chunk past the diagonal)
        for c in (both, cover[0]):
            extra = (c > 0) & ~want
            assert np.all(extra.sum(axis=1) <= 1), ctx
        # the first launch holds what the next step reads: its block row
        # (tile row 0) and its block column [k + b, k + b + 128)
        nxt = np.zeros_like(want)
        nxt[0, :] = True
        nxt[:, 2 * pri_nt: 2 * pri_nt + 2] = True
        assert np.all(cover[1][nxt & want] == 1), ctx
        # and nothing else: the rest launch is disjoint from it
        assert np.all(cover[1][~nxt] == 0), ctx


def test_narrow_tiles_when_a_launch_fills_few_sms(lib):
    # 3 x 3 tiles of 128 fill 9 SMs: narrow (128 x 64) tiles, twice as many
    bn, tiles = plan(lib, 384, 384, 0, 0, 0, 0)
    assert bn == 64 and len(tiles) == 18
    # 128 tiles of 128 fill most of 148 SMs: wide tiles
    bn, tiles = plan(lib, 128 * 16, 128 * 8, 0, 0, 0, 0)
    assert bn == 128 and len(tiles) == 128
    # the same launch on a GPU with twice the SMs goes narrow
    bn, tiles = plan(lib, 128 * 16, 128 * 8, 0, 0, 0, 0, sms=2 * 128)
    assert bn == 64 and len(tiles) == 256


def test_tiles_come_row_by_row(lib):
    bn, tiles = plan(lib, 4096 - 256, 4096, 1, 256, 2, 2)
    order = tiles[:, 0].astype(np.int64) * 10_000 + tiles[:, 1]
    assert np.all(np.diff(order) > 0)


def test_bad_arguments(lib):
    bn = ctypes.c_int(0)
    f = lib.gptq_internal_tgemm_tiles
    assert f(0, 128, 1, 0, 0, 0, 0, SMS, ctypes.byref(bn), None, 0) == -1
    assert f(128, 128, 1, 0, 0, 3, 0, SMS, ctypes.byref(bn), None, 0) == -1
    assert f(128, 128, 1, 0, 0, 0, -1, SMS, ctypes.byref(bn), None, 0) == -1
    assert f(128, 128, 1, 0, 0, 0, 0, 0, ctypes.byref(bn), None, 0) == -1
    assert f(128, 128, 1, 0, 0, 0, 0, SMS, None, None, 0) == -1
    assert f(128, 128, 1, 0, 0, 0, 0, SMS, ctypes.byref(bn), None, 4) == -1
