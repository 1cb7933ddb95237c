"""The C-ABI library loads and exports every symbol include/gptq.h declares;
host-side argument checks and schedules behave as documented.  No GPU."""
import ctypes
import os
import re

import pytest

from post_weight_quantization_31_b300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gptq.h")


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    return re.findall(r"GPTQ_API\s+[\w\s\*]+?\b(gptq_\w+)\s*\(", text)


@pytest.fixture(scope="module")
def lib():
    from post_weight_quantization_31_b300 import build_lib
    build_lib.build()
    return _lib.load()


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for n in ("gptq_hessian_accumulate", "gptq_prepare_hinv", "gptq_quantize_layer",
              "gptq_pack", "gptq_unpack", "gptq_prepare_workspace_size",
              "gptq_quantize_workspace_size", "gptq_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(declared_functions()) == set(_lib.SIGNATURES)


def test_status_strings(lib):
    for code in range(8):
        s = lib.gptq_status_string(code)
        assert isinstance(s, bytes) and len(s) >= 2
    assert lib.gptq_status_string(0) == b"ok"


def test_workspace_sizes_grow(lib):
    a = lib.gptq_prepare_workspace_size(512)
    b = lib.gptq_prepare_workspace_size(4096)
    assert a >= 512 * 512 * 4 and b >= 4096 * 4096 * 4 and b > a
    cfg = _lib.make_config(type("C", (), dict(bits=4, group_size=128, damp_percent=0.01,
                                              blocksize=128, desc_act=0, sym=0)))
    q = lib.gptq_quantize_workspace_size(4096, 4096, ctypes.byref(cfg))
    assert q >= 4096 * 4096 * 4 + 4096 * 128 * 4
    assert lib.gptq_prepare_workspace_size(0) == 0


FAKE = 1 << 20  # a non-null, aligned address that is never dereferenced


def cfg_c(**kw):
    base = dict(bits=4, group_size=128, damp_percent=0.01, blocksize=128, desc_act=0, sym=0)
    base.update(kw)
    return _lib.GptqConfigC(base["bits"], base["group_size"], base["damp_percent"],
                            base["blocksize"], base["desc_act"], base["sym"])


@pytest.mark.parametrize("d_col,n_tok,ldx", [(0, 64, 64), (48, 64, 64), (64, 0, 64),
                                             (64, 64, 60), (64, 100, 100)])
def test_accumulate_rejects_bad_sizes(lib, d_col, n_tok, ldx):
    n = ctypes.c_int64(0)
    assert lib.gptq_hessian_accumulate(FAKE, d_col, n_tok, ldx, 0, FAKE, None, ctypes.byref(n),
                                       None) == 1
    assert n.value == 0


def test_accumulate_rejects_null_and_misaligned(lib):
    assert lib.gptq_hessian_accumulate(None, 64, 64, 64, 0, FAKE, None, None, None) == 1
    assert lib.gptq_hessian_accumulate(FAKE + 2, 64, 64, 64, 0, FAKE, None, None, None) == 1


@pytest.mark.parametrize("d_col,n_tok,ldx,layout", [(64, 100, 56, 1), (64, 100, 60, 1), (64, 40, 64, 2),
                                                    (96, 10, 72, 1), (64, 100, 64, -1)])
def test_accumulate_rejects_bad_token_major_args(lib, d_col, n_tok, ldx, layout):
    """Token-major X [n_tok, d_col] needs ldx >= d_col (a multiple of 8); the
    layout flag is 0 or 1."""
    n = ctypes.c_int64(0)
    assert lib.gptq_hessian_accumulate(FAKE, d_col, n_tok, ldx, layout, FAKE, None, ctypes.byref(n),
                                       None) == 1
    assert n.value == 0


@pytest.mark.parametrize("kw", [dict(bits=5), dict(bits=1), dict(group_size=48),
                                dict(group_size=256), dict(group_size=0), dict(blocksize=48),
                                dict(blocksize=0), dict(blocksize=-32),
                                dict(damp_percent=-0.1), dict(desc_act=2), dict(sym=3),
                                dict(damp_percent=float("nan"))])
def test_prepare_rejects_bad_config(lib, kw):
    c = cfg_c(**kw)
    st = lib.gptq_prepare_hinv(FAKE, None, 512, 1000, ctypes.byref(c), FAKE, FAKE, FAKE,
                               1 << 40, None)
    assert st == 1, kw


def test_prepare_rejects_small_workspace(lib):
    c = cfg_c()
    need = lib.gptq_prepare_workspace_size(512)
    assert lib.gptq_prepare_hinv(FAKE, None, 512, 1000, ctypes.byref(c), FAKE, FAKE, FAKE,
                                 need - 1, None) == 4
    assert lib.gptq_prepare_hinv(FAKE, None, 512, 1000, ctypes.byref(c), FAKE, FAKE, None,
                                 need, None) == 4


def test_quantize_rejects_bad_args(lib):
    c = cfg_c()
    need = lib.gptq_quantize_workspace_size(256, 512, ctypes.byref(c))
    args = [FAKE, 1, 256, 512, FAKE, FAKE, ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE,
            need, None]
    bad = list(args)
    bad[1] = 7  # w_dtype
    assert lib.gptq_quantize_layer(*bad) == 1
    bad = list(args)
    bad[2] = 250  # d_row % 32
    assert lib.gptq_quantize_layer(*bad) == 1
    bad = list(args)
    bad[3] = 500  # d_col % 32
    assert lib.gptq_quantize_layer(*bad) == 1
    bad = list(args)
    bad[12] = need - 256
    assert lib.gptq_quantize_layer(*bad) == 4
    c2 = cfg_c(group_size=96)  # does not divide 512
    bad = list(args)
    bad[6] = ctypes.byref(c2)
    assert lib.gptq_quantize_layer(*bad) == 1


def test_pack_rejects_bad_args(lib):
    assert lib.gptq_pack(FAKE, FAKE, 256, 512, 5, 128, FAKE, FAKE, None) == 1
    assert lib.gptq_pack(FAKE, FAKE, 250, 512, 4, 128, FAKE, FAKE, None) == 1
    assert lib.gptq_pack(FAKE, FAKE, 256, 512, 4, 96, FAKE, FAKE, None) == 1
    assert lib.gptq_unpack(FAKE, FAKE, 256, 500, 4, 128, FAKE, FAKE, None) == 1


def schedule(lib, d, n_tok, grid):
    out = (ctypes.c_int32 * 5)()
    lib.gptq_internal_syrk_schedule(ctypes.c_int64(d), ctypes.c_int64(n_tok), grid, out)
    return dict(zip(("pairs", "full", "rem", "ks", "jobs"), list(out)))


def upper_tile_pairs(d):
    """Tiles of 128 rows x 256 cols that hold some (r, c) with r <= c, counted
    per column block; each column block's tiles are taken two row blocks at a
    time (the two CTAs of a cluster), so a block with c tiles has ceil(c/2)
    pairs.  Returns (tiles, pairs)."""
    tiles = pairs = 0
    for tj in range((d + 255) // 256):
        c = sum(1 for ti in range((d + 127) // 128) if 128 * ti <= 256 * tj + 255)
        tiles += c
        pairs += (c + 1) // 2
    return tiles, pairs


@pytest.mark.parametrize("d", [32, 256, 512, 544, 4096, 5120, 11008, 13824])
def test_syrk_schedule_covers_all_tiles(lib, d):
    s = schedule(lib, d, 262144, 74)
    tiles, pairs = upper_tile_pairs(d)
    assert s["pairs"] == pairs and tiles <= 2 * pairs
    assert s["full"] % 74 == 0 and s["full"] + s["rem"] == s["pairs"]
    assert s["jobs"] == s["full"] + s["rem"] * s["ks"]
    assert s["ks"] >= 1 and (s["rem"] > 0 or s["ks"] == 1)
    # each piece keeps at least 8 slabs of 64 tokens
    assert 262144 // 64 // s["ks"] >= 8


def test_syrk_schedule_small_token_count(lib):
    s = schedule(lib, 512, 2048, 74)
    assert s["ks"] <= 2048 // 64 // 8


def test_dequantize_rejects_bad_args(lib):
    ok = dict(qw=FAKE, qz=FAKE, sc=FAKE, gi=FAKE, d_row=64, d_col=256, bits=4, gs=128, dt=2, out=FAKE)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.gptq_dequantize(a["qw"], a["qz"], a["sc"], a["gi"], a["d_row"], a["d_col"], a["bits"],
                                   a["gs"], a["dt"], a["out"], None)
    assert call(bits=5) == 1
    assert call(d_col=250) == 1
    assert call(gs=96) == 1
    assert call(dt=7) == 1
    assert call(out=FAKE + 8) == 1      # output must be 16-byte aligned
    assert call(qw=0) == 1


def test_dequant_matmul_rejects_bad_args(lib):
    ok = dict(X=FAKE, dt=2, M=16, ldx=256, qw=FAKE, qz=FAKE, sc=FAKE, gi=FAKE, d_row=128, d_col=256,
              bits=4, gs=128, Y=FAKE)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.gptq_dequant_matmul(a["X"], a["dt"], a["M"], a["ldx"], a["qw"], a["qz"], a["sc"],
                                       a["gi"], a["d_row"], a["d_col"], a["bits"], a["gs"], a["Y"], None)
    assert call(dt=0) == 1              # fp32 activations are not a tensor-core operand here
    assert call(M=0) == 1
    assert call(ldx=200) == 1           # ldx < d_col
    assert call(ldx=260) == 1           # ldx % 8 != 0
    assert call(d_col=224) == 1         # d_col % 64 != 0
    assert call(X=FAKE + 8) == 1        # X must be 16-byte aligned
    assert call(gi=FAKE + 4) == 1       # g_idx must be 16-byte aligned
    assert call(sc=FAKE + 4) == 1       # scales must be 16-byte aligned
    assert call(Y=0) == 1


@pytest.mark.parametrize("kw,frac,grid", [(dict(), 0.0, [1.0]), (dict(), 1.5, [1.0]),
                                          (dict(), 0.05, []), (dict(), 0.05, [1.0, -2.0]),
                                          (dict(bits=5), 0.05, [1.0]), (dict(group_size=48), 0.05, [1.0])])
def test_awq_rejects_bad_args(lib, kw, frac, grid):
    c = cfg_c(**kw)
    g = (ctypes.c_float * max(1, len(grid)))(*grid)
    need = lib.gptq_awq_workspace_size(64, 256, max(1, len(grid)))
    st = lib.gptq_awq_search(FAKE, 1, 64, 256, FAKE, FAKE, ctypes.byref(c), frac,
                             ctypes.cast(g, ctypes.c_void_p), len(grid), FAKE, FAKE, FAKE, FAKE, None,
                             FAKE, need, None)
    assert st == 1, (kw, frac, grid)


def test_awq_rejects_missing_diag_and_small_workspace(lib):
    c = cfg_c()
    g = (ctypes.c_float * 2)(1.0, 2.0)
    need = lib.gptq_awq_workspace_size(64, 256, 2)
    args = [FAKE, 1, 64, 256, FAKE, None, ctypes.byref(c), 0.05, ctypes.cast(g, ctypes.c_void_p), 2,
            FAKE, FAKE, FAKE, FAKE, None, FAKE, need, None]
    assert lib.gptq_awq_search(*args) == 1
    args[5] = FAKE
    args[16] = need - 1
    assert lib.gptq_awq_search(*args) == 4
