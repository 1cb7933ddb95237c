// fp32-accurate GEMM on the 5th-generation tensor cores ("3xTF32").
//
//   C[m, n] = alpha * sum_k A[m, k] B[n, k] + beta * C[m, n]
//
// A [M, K] and B [N, K] are row-major (K contiguous, "K-major") and each is
// given as two fp32 arrays hi + lo with hi exactly representable in TF32
// (10-bit mantissa) and lo ~ x - hi; see split_tf32().  The product is
// formed as A_lo B_hi + A_hi B_lo + A_hi B_hi with fp32 accumulation in
// TMEM, which keeps about 2^-21 relative accuracy per product (the dropped
// A_lo B_lo term is ~2^-22).  With `lower`, only elements with
// row_off + m >= col_off + n are written, and tiles entirely above that
// diagonal are skipped.
//
// Requirements: K % 32 == 0 is not needed (TMA zero-fills), but lda, ldb
// (elements) must be multiples of 4 and A/B 16-byte aligned; ldc any.
#pragma once

#include "common.cuh"

namespace gptq {

struct TGemmArgs {
  int M, N, K;
  float alpha, beta;
  float* C;
  int64_t ldc;
  int lower;
  int row_off, col_off;
  // Optional, with lower = 1, alpha = -1, beta = 1: for the elements on the
  // diagonal (row_off + m == col_off + n), the exact rounding error of the
  // update (Knuth two-sum) is added to diag_lo[col_off + n], so that
  // C + diag_lo carries the running diagonal to about twice fp32 precision.
  float* diag_lo = nullptr;
  // Optional tile subsets, for splitting one update into two launches:
  // subset 1 takes the tiles of the first 128 rows (tile row 0) and of the
  // 128 columns [128 pri_nt, 128 pri_nt + 128); subset 2 takes all the
  // others; 0 takes every tile.  The two subsets together are the whole
  // update, each element computed exactly as the single launch computes it.
  int subset = 0;
  int pri_nt = 0;
  // At most this many CTAs (0: one per SM).
  int max_ctas = 0;
};

// hi: x rounded to a TF32 value (10 explicit mantissa bits, ties away);
// lo: x - hi rounded the same way (|x - hi - lo| <= 2^-22 |x|).
__device__ __forceinline__ float round_tf32(float x) {
  const uint32_t u = __float_as_uint(x);
  const float r = __uint_as_float((u + 0x1000u) & 0xFFFFE000u);
  return isfinite(r) ? r : __uint_as_float(u & 0xFFFFE000u);
}
__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
  hi = round_tf32(x);
  // The tensor cores read only the TF32 bits of lo; rounding it here (rather
  // than letting the low bits be dropped) halves what the pair leaves out.
  lo = round_tf32(__fsub_rn(x, hi));
}

// `fault`: the status word the kernel's bounded waits report a timeout in
// (and read to stop early once one has run out).
gptq_status_t launch_tgemm_3xtf32(const float* A_hi, const float* A_lo, int64_t lda,
                                  const float* B_hi, const float* B_lo, int64_t ldb,
                                  const TGemmArgs& args, int* fault, cudaStream_t st);

// Number of 128 x 128 output tiles of the launch's subset (a launch that
// would fill fewer than half the SMs runs 128 x 64 tiles instead, twice as
// many).
int tgemm_tile_count(const TGemmArgs& args);

}  // namespace gptq
