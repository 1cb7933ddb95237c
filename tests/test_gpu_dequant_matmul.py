"""gptq_dequant_matmul against the oracle: Y = X · Wᵀ with W the packed
layer (written by the oracle's packers) dequantized and rounded to X's type.
The kernel sums fp32 products in its own order, so the bar is the rounding
bound of an fp32 sum of K terms plus the split-K additions:
|Y − Y_ref| <= (K + 148)·2⁻²³·Σ_k |X[m][k]·W[n][k]|.  A wrong code, group,
scale or zero moves an output by about one term's size, far above it."""
import numpy as np
import pytest

import oracle as O
from tests.test_gpu_dequant import packed_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from post_weight_quantization_31_b300 import build_lib
    build_lib.build()


TDT = {"fp16": "float16", "bf16": "bfloat16"}


def run_case(M, N, K, bits, gs, act_order, dt, seed, ldx=None):
    import torch
    from post_weight_quantization_31_b300 import api
    codes, zeros, scales, g_idx = packed_case(N, K, bits, gs, act_order, seed)
    rng = np.random.Generator(np.random.PCG64(seed + 1))
    ldx = K if ldx is None else ldx
    Xfull = torch.from_numpy(rng.standard_normal((M, ldx)).astype(np.float32)).to(getattr(torch, TDT[dt]))
    X = Xfull[:, :K]
    qw = torch.from_numpy(O.pack_qweight(codes, bits)).cuda()
    qz = torch.from_numpy(O.pack_qzeros(zeros, bits)).cuda()
    sc = torch.from_numpy(scales).cuda()
    gi = torch.from_numpy(g_idx.astype(np.int32)).cuda()
    Xd = Xfull.cuda()[:, :K]
    Y = api.dequant_matmul(Xd, qw, qz, sc, gi, N, K, bits, gs)
    torch.cuda.synchronize()
    X64 = X.float().numpy().astype(np.float64)
    want = O.dequant_matmul(X64, codes, scales, zeros, g_idx, dt)
    W = O.dequantize_as(codes, scales, zeros, g_idx, dt).astype(np.float64)
    bound = (K + 148) * 2.0 ** -23 * (np.abs(X64) @ np.abs(W).T)
    got = Y.cpu().numpy().astype(np.float64)
    err = np.abs(got - want)
    assert np.all(err <= bound + 1e-30), float((err / (bound + 1e-30)).max())
    return got, want


@pytest.mark.parametrize("dt", ["fp16", "bf16"])
@pytest.mark.parametrize("M,N,K,bits,gs,act", [
    (1, 128, 64, 4, 64, False),          # one slab, one tile, a single activation row
    (16, 256, 1024, 4, 128, False),      # decode batch, split K
    (17, 96, 512, 3, 128, True),         # partial n tile, ragged M, act-order
    (300, 384, 768, 2, 64, False),       # two m tiles (256 + 44)
    (64, 160, 1024, 8, 32, True),        # 8-bit, 32-wide groups, act-order
    (8, 128, 2048, 4, -1, False),        # one group per row
])
def test_dequant_matmul_matches_oracle(M, N, K, bits, gs, act, dt):
    run_case(M, N, K, bits, gs, act, dt, seed=M + N + K + bits)


def test_dequant_matmul_strided_x():
    run_case(5, 128, 256, 4, 128, False, "fp16", seed=8, ldx=264)


def test_dequant_matmul_many_groups():
    """1280 groups of 32: the scale table does not fit in shared memory and
    scales and zeros are read from global memory."""
    run_case(4, 128, 40960, 4, 32, True, "bf16", seed=6)


def test_dequant_matmul_full_size_sampled():
    """A 4096 x 4096 4-bit layer (packed on the GPU) times a 16-row decode
    batch and a 4096-row prefill batch; sampled output features checked
    against the oracle one by one."""
    import torch
    from post_weight_quantization_31_b300 import api
    N = K = 4096
    bits, gs = 4, 128
    rng = np.random.Generator(np.random.PCG64(31))
    G = K // gs
    codes = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    zeros = rng.integers(0, 16, size=(G, N), dtype=np.uint8)
    scales = rng.uniform(1e-3, 2e-2, size=(G, N)).astype(np.float32)
    g_idx = O.group_index(np.arange(K), gs)
    qw, qz = api.pack(torch.from_numpy(codes).cuda(), torch.from_numpy(zeros).cuda(), bits, gs)
    sc = torch.from_numpy(scales).cuda()
    gi = torch.from_numpy(g_idx.astype(np.int32)).cuda()
    ns = np.sort(rng.choice(N, size=24, replace=False))
    for M in (16, 4096):
        X = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).half()
        Y = api.dequant_matmul(X.cuda(), qw, qz, sc, gi, N, K, bits, gs)
        torch.cuda.synchronize()
        ms = np.sort(rng.choice(M, size=min(M, 16), replace=False))
        X64 = X.float().numpy().astype(np.float64)[ms]
        c, z = codes[ns].astype(np.int64), zeros[:, ns].astype(np.int64)
        want = O.dequant_matmul(X64, c, scales[:, ns], z, g_idx, "fp16")
        W = O.dequantize_as(c, scales[:, ns], z, g_idx, "fp16").astype(np.float64)
        bound = (K + 148) * 2.0 ** -23 * (np.abs(X64) @ np.abs(W).T)
        got = Y.cpu().numpy()[np.ix_(ms, ns)].astype(np.float64)
        assert np.all(np.abs(got - want) <= bound), M
