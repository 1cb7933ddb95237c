// fp32 FFMA tile GEMM used by the blocked Cholesky, the triangular inverse
// and the trailing lazy-batch update:
//
//   C[m, n] = alpha * sum_k opA[m, k] * opB[k, n] + beta * C[m, n]
//
// A is row-major [M, K] (lda).  B is row-major [K, N] (ldb) or, with
// B_NK, given as row-major [N, K] (ldb) and used transposed.  Optional
// triangular masks treat entries outside a lower triangle as exact zeros
// (the stored values there are ignored, whatever they are):
//   A_LOWER:    opA[m, k] = 0 for k > m
//   B_LOWER:    opB[k, n] = 0 for n > k
// and shorten the K loop accordingly.
//
// One CTA computes a 128 x 128 tile with 256 threads (8 x 8 outputs each),
// K in slabs of 8 through double-buffered shared memory.  M, N and K must
// be multiples of 4 and all pointers/leading dimensions 16-byte aligned
// (float4 loads); partial tiles are handled.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gptq {

constexpr int GM = 128;
constexpr int GN = 128;
constexpr int GK = 8;
constexpr int GEMM_THREADS = 256;

struct GemmArgs {
  int M, N, K;
  float alpha, beta;
  const float* A;
  int64_t lda;
  const float* B;
  int64_t ldb;
  float* C;
  int64_t ldc;
};

struct GemmSmem {
  float As[2][GK][GM];
  float Bs[2][GK][GN];
};

template <bool B_NK, bool A_LOWER, bool B_LOWER>
__device__ __forceinline__ void gemm_load_slab(const GemmArgs& g, int m0, int n0, int k0, float4& ra,
                                               float4& rb) {
  const int t = threadIdx.x;
  {  // A: 128 rows x 8 k, one float4 along k per thread
    const int m = t >> 1, kq = (t & 1) * 4;
    const int gm = m0 + m, gk = k0 + kq;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (gm < g.M && gk < g.K) v = *reinterpret_cast<const float4*>(g.A + gm * g.lda + gk);
    if (A_LOWER) {
      if (gk + 0 > gm) v.x = 0.f;
      if (gk + 1 > gm) v.y = 0.f;
      if (gk + 2 > gm) v.z = 0.f;
      if (gk + 3 > gm) v.w = 0.f;
    }
    ra = v;
  }
  if (!B_NK) {  // B [K, N]: 8 k x 128 n, one float4 along n per thread
    const int k = t >> 5, nq = (t & 31) * 4;
    const int gk = k0 + k, gn = n0 + nq;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (gk < g.K && gn < g.N) v = *reinterpret_cast<const float4*>(g.B + gk * g.ldb + gn);
    if (B_LOWER) {
      if (gn + 0 > gk) v.x = 0.f;
      if (gn + 1 > gk) v.y = 0.f;
      if (gn + 2 > gk) v.z = 0.f;
      if (gn + 3 > gk) v.w = 0.f;
    }
    rb = v;
  } else {  // B given as [N, K]: one float4 along k per thread
    const int n = t >> 1, kq = (t & 1) * 4;
    const int gn = n0 + n, gk = k0 + kq;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (gn < g.N && gk < g.K) v = *reinterpret_cast<const float4*>(g.B + gn * g.ldb + gk);
    if (B_LOWER) {
      if (gn > gk + 0) v.x = 0.f;
      if (gn > gk + 1) v.y = 0.f;
      if (gn > gk + 2) v.z = 0.f;
      if (gn > gk + 3) v.w = 0.f;
    }
    rb = v;
  }
}

template <bool B_NK>
__device__ __forceinline__ void gemm_store_slab(GemmSmem& s, int buf, const float4& ra, const float4& rb) {
  const int t = threadIdx.x;
  {
    const int m = t >> 1, kq = (t & 1) * 4;
    s.As[buf][kq + 0][m] = ra.x;
    s.As[buf][kq + 1][m] = ra.y;
    s.As[buf][kq + 2][m] = ra.z;
    s.As[buf][kq + 3][m] = ra.w;
  }
  if (!B_NK) {
    const int k = t >> 5, nq = (t & 31) * 4;
    *reinterpret_cast<float4*>(&s.Bs[buf][k][nq]) = rb;
  } else {
    const int n = t >> 1, kq = (t & 1) * 4;
    s.Bs[buf][kq + 0][n] = rb.x;
    s.Bs[buf][kq + 1][n] = rb.y;
    s.Bs[buf][kq + 2][n] = rb.z;
    s.Bs[buf][kq + 3][n] = rb.w;
  }
}

// Computes the tile at (m0, n0).  `lower_only` skips tiles entirely above
// the diagonal of C (n0 > m0 + GM - 1), for symmetric updates.
template <bool B_NK, bool A_LOWER, bool B_LOWER>
__device__ void gemm_tile(const GemmArgs& g, int m0, int n0, GemmSmem& s) {
  if (m0 >= g.M || n0 >= g.N) return;
  int k_begin = 0, k_end = g.K;
  if (A_LOWER) k_end = min(k_end, m0 + GM);          // opA[m, k] = 0 for k > m
  if (B_LOWER) k_begin = (n0 / GK) * GK;             // opB[k, n] = 0 for k < n
  const int t = threadIdx.x;
  const int tx = t & 15, ty = t >> 4;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  if (k_begin < k_end) {
    float4 ra, rb;
    gemm_load_slab<B_NK, A_LOWER, B_LOWER>(g, m0, n0, k_begin, ra, rb);
    gemm_store_slab<B_NK>(s, 0, ra, rb);
    __syncthreads();
    int buf = 0;
    for (int k0 = k_begin; k0 < k_end; k0 += GK) {
      const bool more = k0 + GK < k_end;
      if (more) gemm_load_slab<B_NK, A_LOWER, B_LOWER>(g, m0, n0, k0 + GK, ra, rb);
#pragma unroll
      for (int kk = 0; kk < GK; ++kk) {
        const float4 a0 = *reinterpret_cast<const float4*>(&s.As[buf][kk][ty * 4]);
        const float4 a1 = *reinterpret_cast<const float4*>(&s.As[buf][kk][64 + ty * 4]);
        const float4 b0 = *reinterpret_cast<const float4*>(&s.Bs[buf][kk][tx * 4]);
        const float4 b1 = *reinterpret_cast<const float4*>(&s.Bs[buf][kk][64 + tx * 4]);
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
      if (more) {
        gemm_store_slab<B_NK>(s, buf ^ 1, ra, rb);
        __syncthreads();
        buf ^= 1;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    if (m >= g.M) continue;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int n = n0 + h * 64 + tx * 4;
      if (n >= g.N) continue;
      float* cp = g.C + m * g.ldc + n;
      float4 out = make_float4(g.alpha * acc[i][h * 4 + 0], g.alpha * acc[i][h * 4 + 1],
                               g.alpha * acc[i][h * 4 + 2], g.alpha * acc[i][h * 4 + 3]);
      if (g.beta != 0.f) {
        const float4 c = *reinterpret_cast<const float4*>(cp);
        out.x = fmaf(g.beta, c.x, out.x);
        out.y = fmaf(g.beta, c.y, out.y);
        out.z = fmaf(g.beta, c.z, out.z);
        out.w = fmaf(g.beta, c.w, out.w);
      }
      *reinterpret_cast<float4*>(cp) = out;
    }
  }
}

}  // namespace gptq
