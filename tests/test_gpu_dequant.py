"""gptq_dequantize against the oracle: packed layer (written by the oracle's
own packers) -> dense weights in the original column order.  Both sides form
scale * (code - zero) as one fp32 product and round it once to the storage
type, so the comparison is bit-exact for fp32, fp16 and bf16."""
import numpy as np
import pytest

import oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from post_weight_quantization_31_b300 import build_lib
    build_lib.build()


DT = {"fp32": "float32", "fp16": "float16", "bf16": "bfloat16"}


def packed_case(d_row, d_col, bits, gs, act_order, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    codes = rng.integers(0, 1 << bits, size=(d_row, d_col))
    G = 1 if gs == -1 else -(-d_col // gs)
    zeros = rng.integers(0, 1 << bits, size=(G, d_row))
    scales = (rng.uniform(0.5, 2.0, size=(G, d_row)) * 10.0 ** rng.integers(-4, 1, size=(G, d_row))
              ).astype(np.float32)
    perm = rng.permutation(d_col) if act_order else np.arange(d_col)
    g_idx = O.group_index(perm, gs)
    return codes, zeros, scales, g_idx


def gpu_dequant(codes, zeros, scales, g_idx, bits, gs, dt):
    import torch
    from post_weight_quantization_31_b300 import api
    d_row, d_col = codes.shape
    qw = torch.from_numpy(O.pack_qweight(codes, bits)).cuda()
    qz = torch.from_numpy(O.pack_qzeros(zeros, bits)).cuda()
    sc = torch.from_numpy(scales).cuda()
    gi = torch.from_numpy(g_idx.astype(np.int32)).cuda()
    out = api.dequantize(qw, qz, sc, gi, d_row, d_col, bits, gs, dtype=getattr(torch, DT[dt]))
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


@pytest.mark.parametrize("dt", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("bits,gs,act_order,d_col", [(4, 128, False, 1152), (4, 128, True, 1152),
                                                     (3, 128, True, 1152), (2, 64, False, 1152),
                                                     (8, 32, True, 800), (4, -1, False, 800),
                                                     (3, -1, True, 1152)])
def test_dequantize_bit_exact(bits, gs, act_order, d_col, dt):
    # 1152 columns: 4 full 256-column chunks and a 128-column tail; 800: a
    # 32-column tail; 96 rows: 3 row blocks
    d_row = 96
    codes, zeros, scales, g_idx = packed_case(d_row, d_col, bits, gs, act_order, seed=bits * 7 + d_row)
    got = gpu_dequant(codes, zeros, scales, g_idx, bits, gs, dt)
    want = O.dequantize_as(codes, scales, zeros, g_idx, dt)
    assert np.array_equal(got, want)


def test_dequantize_smallest_shape():
    codes, zeros, scales, g_idx = packed_case(32, 32, 3, 32, False, seed=3)
    got = gpu_dequant(codes, zeros, scales, g_idx, 3, 32, "fp32")
    assert np.array_equal(got, O.dequantize_as(codes, scales, zeros, g_idx, "fp32"))


def test_dequantize_many_groups():
    """More groups than the shared-memory scale table holds (1280 groups of
    32): scales and zeros are read from global memory."""
    codes, zeros, scales, g_idx = packed_case(32, 40960, 4, 32, True, seed=5)
    got = gpu_dequant(codes, zeros, scales, g_idx, 4, 32, "fp16")
    assert np.array_equal(got, O.dequantize_as(codes, scales, zeros, g_idx, "fp16"))


def test_dequantize_out_of_range_g_idx_is_clamped():
    codes, zeros, scales, g_idx = packed_case(64, 512, 4, 128, False, seed=9)
    bad = g_idx.copy()
    bad[:7] = -3
    bad[-5:] = 99
    got = gpu_dequant(codes, zeros, scales, bad, 4, 128, "fp32")
    assert np.array_equal(got, O.dequantize_as(codes, scales, zeros, np.clip(bad, 0, 3), "fp32"))


def test_dequantize_full_size_sampled_rows():
    """A 4096 x 11008 4-bit act-order layer, packed on the GPU; sampled rows
    are unpacked and dequantized one by one by the oracle."""
    import torch
    from post_weight_quantization_31_b300 import api
    d_row, d_col, bits, gs = 4096, 11008, 4, 128
    rng = np.random.Generator(np.random.PCG64(21))
    G = d_col // gs
    codes = torch.from_numpy(rng.integers(0, 16, size=(d_row, d_col), dtype=np.uint8)).cuda()
    zeros = torch.from_numpy(rng.integers(0, 16, size=(G, d_row), dtype=np.uint8)).cuda()
    scales_h = rng.uniform(1e-3, 2e-2, size=(G, d_row)).astype(np.float32)
    g_idx_h = O.group_index(rng.permutation(d_col), gs)
    qw, qz = api.pack(codes, zeros, bits, gs)
    out = api.dequantize(qw, qz, torch.from_numpy(scales_h).cuda(),
                         torch.from_numpy(g_idx_h.astype(np.int32)).cuda(), d_row, d_col, bits, gs,
                         dtype=torch.float16)
    torch.cuda.synchronize()
    rows = np.sort(rng.choice(d_row, size=16, replace=False))
    got = out[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    codes_h = codes.cpu().numpy().astype(np.int64)          # the generator's codes
    zeros_h = zeros.cpu().numpy().astype(np.int64)
    want = O.dequantize_as(codes_h[rows], scales_h[:, rows], zeros_h[:, rows], g_idx_h, "fp16")
    assert np.array_equal(got, want)
    # the GPU packing of the sampled rows, against the oracle's packer
    qw_h = qw.cpu().numpy()
    assert np.array_equal(qw_h[:, rows], O.pack_qweight(codes_h[rows], bits))


def test_container_round_trip_of_a_solved_layer(tmp_path):
    """A layer solved on the GPU, saved with quantize_config.json + safetensors,
    loaded back and dequantized: the same dense weights as before saving."""
    import torch
    from post_weight_quantization_31_b300 import api, container
    from post_weight_quantization_31_b300 import workloads as wl
    cfg = wl.QuantConfig(bits=4, group_size=64, desc_act=True)
    d_row, d_col = 64, 256
    W = torch.from_numpy(wl.make_weight(d_row, d_col, seed=3)).cuda()
    X = torch.from_numpy(wl.make_activations(d_col, 1024, seed=4)).cuda()
    solver = api.LayerSolver(d_row, d_col, cfg)
    solver.reset()
    res = solver.solve(W, X)
    before = api.dequantize(res.qweight, res.qzeros, res.scales, res.g_idx, d_row, d_col, 4, 64,
                            dtype=torch.float32)
    container.save_quantized(str(tmp_path), {"layer": res}, cfg)
    layers, cfg2 = container.load_quantized(str(tmp_path))
    assert cfg2 == cfg
    L = {k: torch.from_numpy(v).cuda() for k, v in layers["layer"].items()}
    after = api.dequantize(L["qweight"], L["qzeros"], L["scales"], L["g_idx"], d_row, d_col, 4, 64,
                           dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(before, after)
