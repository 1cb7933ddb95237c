"""The layer solve spread over several GPUs, one process per GPU.

Two data-parallel layouts of one layer (GPTQ practical guide,
m.lqnn.cn/news/117696, §2.2: a 175B model is quantized on four A100s), and
the plain one of whole layers per GPU:

  tokens  step a1 is a sum over calibration tokens, S = sum_t x_t x_t^T, so
          each rank accumulates S over its own contiguous share of the
          tokens and one all-reduce (sum) of S -- with the fp64 diagonal and
          the token count -- gives every rank the Hessian of all tokens.
  rows    in steps a3-a5 the rows of W never interact: the compensation of
          a quantized weight only moves along its own row, through U.  So one
          rank prepares U and the column order from the shared S, broadcasts
          them once, and every rank quantizes and packs its own block of
          rows.  The packed layer is the column-wise concatenation of the
          ranks' qweight / qzeros blocks and the row-wise one of their scales.
  layers  independent layers per GPU need no exchange at all (the benchmark's
          default for several GPUs).

The functions below do the partitioning and the collectives; the arithmetic
is passed in (`accumulate`, `prepare`, `quantize`), so the same orchestration
runs the CUDA library on GPUs over NCCL and, in the tests, a CPU reference
over gloo.  Collectives are torch.distributed calls on the default group
unless `group` is given.
"""
from __future__ import annotations

import dataclasses
from typing import Callable


def split_range(n: int, parts: int, index: int, align: int = 1) -> tuple[int, int]:
    """[a, b) of share `index` when n items are cut into `parts` contiguous
    shares whose boundaries are multiples of `align` (except the end n).
    Shares differ by at most one `align` unit; some may be empty."""
    if parts < 1 or not 0 <= index < parts or align < 1 or n < 0:
        raise ValueError("bad split")
    units = -(-n // align)
    a = min(n, (units * index // parts) * align)
    b = min(n, (units * (index + 1) // parts) * align)
    return a, b


def token_range(n_tok: int, world: int, rank: int) -> tuple[int, int]:
    """This rank's calibration tokens (64-token units, one tensor-core slab)."""
    return split_range(n_tok, world, rank, align=64)


def row_range(d_row: int, world: int, rank: int) -> tuple[int, int]:
    """This rank's rows of W, in 32-row units: the zero points are packed as
    a bit stream along the rows, 32 rows to `bits` words, so 32-row shards
    pack into whole words that concatenate into the layer's qzeros (and the
    library wants d_row % 32 == 0)."""
    if d_row % 32:
        raise ValueError("d_row must be a multiple of 32")
    return split_range(d_row, world, rank, align=32)


def allreduce_hessian(dist, S, diag, n_local: int, group=None) -> int:
    """Sums the ranks' partial Hessians in place (S and, if given, the fp64
    diagonal) and returns the total token count."""
    import torch
    dist.all_reduce(S, op=dist.ReduceOp.SUM, group=group)
    if diag is not None:
        dist.all_reduce(diag, op=dist.ReduceOp.SUM, group=group)
    n = torch.tensor([int(n_local)], dtype=torch.int64, device=S.device)
    dist.all_reduce(n, op=dist.ReduceOp.SUM, group=group)
    return int(n.item())


def broadcast_factor(dist, U, perm, src: int = 0, group=None) -> None:
    """U and the column order from rank `src` to every rank (in place)."""
    dist.broadcast(U, src=src, group=group)
    dist.broadcast(perm, src=src, group=group)


@dataclasses.dataclass
class ShardedResult:
    rows: tuple[int, int]      # this rank's rows [r0, r1) of W
    n_seen: int                # tokens over all ranks
    out: object                # whatever `quantize` returned for the rows


def sharded_layer_solve(dist, rank: int, *, X_local, W_rows, rows: tuple[int, int], S, diag, U,
                        perm, accumulate: Callable, prepare: Callable, quantize: Callable,
                        src: int = 0, group=None) -> ShardedResult:
    """Both layouts in one solve: tokens for the Hessian, rows for the rest.

    X_local   this rank's tokens (token_range), in whatever form `accumulate`
              takes; W_rows this rank's rows [r0, r1) = `rows` (row_range)
              of W.
    S, diag   this rank's zeroed Hessian buffers (diag may be None); U, perm
              buffers for the factor and the order, the same shapes on every
              rank.
    accumulate(X_local, S, diag) -> tokens added;  prepare(S, diag, n, U,
    perm) fills U and perm (called on rank `src` only);  quantize(W_rows, U,
    perm) -> the rows' result.
    """
    n_local = accumulate(X_local, S, diag)
    n = allreduce_hessian(dist, S, diag, n_local, group=group)
    if rank == src:
        prepare(S, diag, n, U, perm)
    broadcast_factor(dist, U, perm, src=src, group=group)
    return ShardedResult(rows=tuple(rows), n_seen=n, out=quantize(W_rows, U, perm))
