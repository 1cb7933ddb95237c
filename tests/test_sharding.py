"""The multi-GPU layouts of the layer solve, checked on CPU with gloo ranks
(spawned processes) and the oracle as the arithmetic:

  tokens  the ranks' partial Hessians, summed by one all-reduce, equal the
          Hessian of all tokens;
  rows    every rank quantizes its own rows with the factor one rank
          computed and broadcast; together the ranks' codes, scales and
          zero points equal the single-process solve of the whole layer
          (rows are independent: pin I3).
"""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from post_weight_quantization_31_b300 import sharding  # noqa: E402


@pytest.mark.parametrize("n,parts,align", [(262144, 8, 64), (1000, 3, 64), (100, 4, 64),
                                           (4096, 3, 32), (96, 4, 32), (0, 2, 32)])
def test_split_range_tiles_the_range(n, parts, align):
    spans = [sharding.split_range(n, parts, i, align) for i in range(parts)]
    assert spans[0][0] == 0 and spans[-1][1] == n
    for (a, b), (c, d) in zip(spans, spans[1:]):
        assert b == c
    for a, b in spans:
        assert a <= b and a % align == 0 and (b % align == 0 or b == n)
    sizes = [(b - a + align - 1) // align for a, b in spans]
    assert max(sizes) - min(sizes) <= 1


def _inputs():
    from post_weight_quantization_31_b300 import workloads as wl
    X = wl.make_activations(192, 1000, seed=41, n_outliers=3, outlier_scale=20.0)
    W = wl.make_weight(96, 192, seed=42, dtype="bf16")
    cfg = wl.QuantConfig(bits=4, group_size=64, damp_percent=0.01, blocksize=128,
                         desc_act=True, sym=False)
    return X, W, cfg


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist

    import oracle as O
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        X, W, cfg = _inputs()
        d_row, d_col = W.shape
        t0, t1 = sharding.token_range(X.shape[1], world, rank)
        r0, r1 = sharding.row_range(d_row, world, rank)
        S = torch.zeros((d_col, d_col), dtype=torch.float64)
        diag = torch.zeros(d_col, dtype=torch.float64)
        U = torch.zeros((d_col, d_col), dtype=torch.float64)
        perm = torch.zeros(d_col, dtype=torch.int64)
        calls = {"prepare": 0}

        def accumulate(Xl, S_, diag_):
            S_ += torch.from_numpy(O.hessian_sum(Xl))
            diag_ += torch.from_numpy(O.hessian_diag(Xl))
            return Xl.shape[1]

        def prepare(S_, diag_, n, U_, perm_):
            calls["prepare"] += 1
            p, _Hp, Uo = O.prepare(S_.numpy(), n, cfg)
            U_.copy_(torch.from_numpy(Uo))
            perm_.copy_(torch.from_numpy(p))

        def quantize(Wr, U_, perm_):
            p = perm_.numpy()
            codes_p, scales, zeros, _Q = O.column_loop(Wr.astype(np.float64)[:, p], U_.numpy(), cfg)
            codes = np.empty_like(codes_p)
            codes[:, p] = codes_p
            return codes, scales, zeros

        res = sharding.sharded_layer_solve(dist, rank, X_local=X[:, t0:t1], W_rows=W[r0:r1],
                                           rows=(r0, r1), S=S, diag=diag, U=U, perm=perm,
                                           accumulate=accumulate, prepare=prepare,
                                           quantize=quantize)
        codes, scales, zeros = res.out
        q.put((rank, (t0, t1), res.rows, res.n_seen, calls["prepare"], S.numpy(), diag.numpy(),
               perm.numpy(), codes, scales, zeros))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_token_and_row_sharded_solve_equals_single_process(world):
    import torch.multiprocessing as mp

    import oracle as O
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29700 + os.getpid() % 200 + 10 * world
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in procs), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    X, W, cfg = _inputs()
    S_full = O.hessian_sum(X)
    full = O.quantize_layer(W, S_full, X.shape[1], cfg)
    # tokens: disjoint shares covering every token; the summed Hessian
    assert res[0][1][0] == 0 and res[-1][1][1] == X.shape[1]
    assert all(a[1][1] == b[1][0] for a, b in zip(res, res[1:]))
    for r in res:
        assert r[3] == X.shape[1]
        np.testing.assert_allclose(r[5], S_full, rtol=1e-12, atol=1e-9)
        np.testing.assert_allclose(r[6], np.diag(S_full), rtol=1e-12)
        assert np.array_equal(r[7], full.perm)
    # the factor was computed once
    assert [r[4] for r in res] == [1] + [0] * (world - 1)
    # rows: together the ranks' codes, scales and zeros are the full solve's
    codes = np.concatenate([r[8] for r in res], axis=0)
    scales = np.concatenate([r[9] for r in res], axis=1)
    zeros = np.concatenate([r[10] for r in res], axis=1)
    assert [r[2] for r in res][0][0] == 0 and res[-1][2][1] == W.shape[0]
    assert np.array_equal(codes, full.codes)
    assert np.array_equal(scales, full.scales)
    assert np.array_equal(zeros, full.zeros)
    # and the row shards pack into whole words of the layer's packed zeros
    parts = [O.pack_qzeros(r[10], cfg.bits) for r in res]
    assert np.array_equal(np.concatenate(parts, axis=1), O.pack_qzeros(full.zeros, cfg.bits))
