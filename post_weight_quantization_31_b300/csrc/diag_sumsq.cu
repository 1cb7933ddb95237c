// Exact-to-rounding diagonal of S = X X^T in fp64: diag[i] += sum_t X[i,t]^2.
//
// The act-order column order ([G] GPTQ practical guide,
// m.lqnn.cn/news/117696, §2.2 and §3.3 desc_act: columns sorted by the
// Hessian diagonal, large first) is an integer decision taken from these
// sums, so they are kept far more accurate than the fp32 tensor-core sums
// of S: each square of an fp16 value is exact in fp32, and the sum is kept
// as an unevaluated pair of fp32 numbers (hi + lo, renormalized after every
// addition with error-free transformations), giving about 2^-44 relative
// error per thread's partial sum.  Partials are combined in fp64 (warp
// shuffles, then one fp64 atomic per block).  B300's fp64 rate is low, so
// the per-element work stays on the fp32 pipes.
#include <cuda_fp16.h>

#include "common.cuh"

namespace gptq {
namespace {

constexpr int DS_THREADS = 256;
constexpr int DS_VEC = 8;                                  // fp16 per 16-byte load
constexpr int DS_ITERS = 8;
constexpr int DS_CHUNK = DS_THREADS * DS_VEC * DS_ITERS;   // tokens per block

struct DF {
  float hi, lo;
};

__device__ __forceinline__ void df_add(DF& a, float v) {
  // Two-sum of hi and v, fold in lo, then fast renormalization.
  const float s = __fadd_rn(a.hi, v);
  const float bb = __fsub_rn(s, a.hi);
  const float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(v, bb));
  const float t = __fadd_rn(e, a.lo);
  a.hi = __fadd_rn(s, t);
  a.lo = __fsub_rn(t, __fsub_rn(a.hi, s));
}

__global__ void __launch_bounds__(DS_THREADS)
    diag_sumsq_kernel(const __half* __restrict__ X, int64_t n_tok, int64_t ldx, double* __restrict__ diag) {
  const int r = blockIdx.x;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * DS_CHUNK;
  const __half* row = X + static_cast<int64_t>(r) * ldx;
  DF acc{0.f, 0.f};
#pragma unroll 2
  for (int it = 0; it < DS_ITERS; ++it) {
    const int64_t t = t0 + (static_cast<int64_t>(it) * DS_THREADS + threadIdx.x) * DS_VEC;
    if (t + DS_VEC <= n_tok) {
      const uint4 u = *reinterpret_cast<const uint4*>(row + t);
      const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(h[k]);
        df_add(acc, __fmul_rn(f.x, f.x));
        df_add(acc, __fmul_rn(f.y, f.y));
      }
    } else if (t < n_tok) {
      for (int64_t k = t; k < n_tok; ++k) {
        const float f = __half2float(row[k]);
        df_add(acc, __fmul_rn(f, f));
      }
    }
  }
  double v = static_cast<double>(acc.hi) + static_cast<double>(acc.lo);
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __shared__ double red[DS_THREADS / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int w = 0; w < DS_THREADS / 32; ++w) tot += red[w];
    atomicAdd(diag + r, tot);
  }
}

// Token-major X [n_tok][ldx] (channels contiguous): each thread owns 8
// consecutive channels (one 16-byte load per token, a warp covers 256
// channels of a token row), the 8 warps of a block take interleaved tokens
// of the block's chunk, and the warps' partials are combined in fp64.
constexpr int DT_WARPS = 8;
constexpr int DT_TOK = 2048;   // tokens per block

__global__ void __launch_bounds__(DT_WARPS * 32)
    diag_sumsq_tokmajor_kernel(const __half* __restrict__ X, int64_t d, int64_t n_tok, int64_t ldx,
                               double* __restrict__ diag) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 256 + lane * 8;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * DT_TOK;
  const int64_t t1 = t0 + DT_TOK < n_tok ? t0 + DT_TOK : n_tok;
  DF acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = DF{0.f, 0.f};
  if (c0 < d) {  // d is a multiple of 8: a thread's 8 channels are all in range or all out
    for (int64_t t = t0 + warp; t < t1; t += DT_WARPS) {
      const uint4 u = *reinterpret_cast<const uint4*>(X + t * ldx + c0);
      const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(h[k]);
        df_add(acc[2 * k], __fmul_rn(f.x, f.x));
        df_add(acc[2 * k + 1], __fmul_rn(f.y, f.y));
      }
    }
  }
  __shared__ double red[DT_WARPS][256];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    red[warp][lane * 8 + k] = static_cast<double>(acc[k].hi) + static_cast<double>(acc[k].lo);
  __syncthreads();
  const int64_t c = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  if (c < d) {
    double tot = 0.0;
#pragma unroll
    for (int w = 0; w < DT_WARPS; ++w) tot += red[w][threadIdx.x];
    atomicAdd(diag + c, tot);
  }
}

}  // namespace

gptq_status_t launch_diag_sumsq(const void* X, int64_t d, int64_t n_tok, int64_t ldx, bool tok_major,
                                double* diag, cudaStream_t st) {
  if (tok_major) {
    dim3 grid(static_cast<unsigned>((d + 255) / 256), static_cast<unsigned>((n_tok + DT_TOK - 1) / DT_TOK));
    diag_sumsq_tokmajor_kernel<<<grid, DT_WARPS * 32, 0, st>>>(static_cast<const __half*>(X), d, n_tok,
                                                                ldx, diag);
  } else {
    dim3 grid(static_cast<unsigned>(d), static_cast<unsigned>((n_tok + DS_CHUNK - 1) / DS_CHUNK));
    diag_sumsq_kernel<<<grid, DS_THREADS, 0, st>>>(static_cast<const __half*>(X), n_tok, ldx, diag);
  }
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

}  // namespace gptq
