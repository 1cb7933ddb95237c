// AWQ scale search (activation-aware weight scaling), the second workload.
//
// Sources:
//   "GPTQ/AWQ量化导出：让大模型在消费级显卡上跑起来", GPTQ/AWQ comparison: the
//     RMS of each channel's activations over the calibration data selects
//     the most active top-k% (5% by default), which get a larger scale.
//   "大模型压缩量化技术：GPTQ 与 AWQ 原理详解 + Python 实战教程", §四: the weights
//     of those channels are multiplied by s > 1 before quantization, the
//     matching activations are divided by s at inference, and the best s is
//     found from forward statistics alone.
// Readings (the same as the CPU oracle's): the statistic is per input
// channel of W, RMS = sqrt(sum_t x^2 / n) (taken from the fp64 sums of
// squares that gptq_hessian_accumulate produces); the salient set is the
// ceil(frac d_col) largest, ties to the lower index; one factor s for all of
// them, chosen among the caller's candidates to minimise the layer output
// error tr(D S D^T), D = W - W_hat, ties to the earlier candidate; the
// quantizer is the GPTQ grid (round to nearest, group-wise, natural column
// order) applied to W diag(t), and W_hat = dequant / t.
//
// Per candidate: one RTN pass over W diag(t) (a warp per row and group, the
// group's min/max by shuffles, codes decided as in the column loop), D as a
// TF32 hi/lo pair; E = D S on the tensor cores (3xTF32, the same GEMM as the
// solver's updates); the error as sum(E .* D) in fp64.  The choice and the
// final quantization run on the device, so the call never waits for the GPU.
#include <cmath>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "tgemm.cuh"

namespace gptq {
namespace {

template <typename T>
__device__ __forceinline__ float awq_f32(T v);
template <>
__device__ __forceinline__ float awq_f32<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float awq_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
template <>
__device__ __forceinline__ float awq_f32<__half>(__half v) {
  return __half2float(v);
}

// The grid of one group of the scaled weights (the column loop's grid).
struct AGrid {
  float s, span, rsp, z;
};

__device__ __forceinline__ float awq_div(float x, const AGrid& g) {
  const float q0 = x * g.rsp;
  const float res = fmaf(-q0, g.span, x);
  return fmaf(res, g.rsp, q0);
}

__device__ __forceinline__ AGrid awq_grid(float xmin, float xmax, float maxq, int sym) {
  xmin = fminf(xmin, 0.f);
  xmax = fmaxf(xmax, 0.f);
  AGrid g;
  float neg_xmin;
  if (sym) {
    float a = fmaxf(-xmin, xmax);
    if (a == 0.f) a = 1.f;
    g.span = 2.f * a;
    neg_xmin = a;
  } else {
    if (xmin == xmax) {
      xmin = -1.f;
      xmax = 1.f;
    }
    g.span = xmax - xmin;
    neg_xmin = -xmin;
  }
  g.s = g.span / maxq;
  g.rsp = 1.f / g.span;
  g.z = sym ? 0.5f * (maxq + 1.f) : rintf(maxq * awq_div(neg_xmin, g));
  return g;
}

// salient[c] = 1 for the k channels with the largest sum of squares (ties:
// lower index first), else 0.  rank(c) = #{j : v_j > v_c} + #{j < c : v_j == v_c}.
__global__ void awq_salient_kernel(const double* __restrict__ diag, int d, int k,
                                   float* __restrict__ salient) {
  __shared__ double tile[1024];
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  const double vc = c < d ? diag[c] : 0.0;
  int rank = 0;
  for (int base = 0; base < d; base += 1024) {
    const int n = min(1024, d - base);
    __syncthreads();
    for (int t = threadIdx.x; t < n; t += blockDim.x) tile[t] = diag[base + t];
    __syncthreads();
    if (c < d)
      for (int t = 0; t < n; ++t) rank += (tile[t] > vc) | ((tile[t] == vc) & (base + t < c));
  }
  if (c < d) salient[c] = rank < k ? 1.f : 0.f;
}

// RTN of W diag(t), t = 1 + salient (factor - 1), one warp per (row, group).
// Search pass (D_hi != null): D = W - dequant / t as a TF32 hi/lo pair.
// Final pass (codes != null): codes, scales, zeros of the scaled weights and
// t itself (written by the warps of row 0).
template <typename T>
__global__ void awq_rtn_kernel(const T* __restrict__ W, int d_row, int d_col, int gs_cols,
                               const float* __restrict__ salient, const float* __restrict__ factor,
                               float maxq, int sym, float* __restrict__ D_hi, float* __restrict__ D_lo,
                               uint8_t* __restrict__ codes, float* __restrict__ scales,
                               uint8_t* __restrict__ zeros, float* __restrict__ t_out) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.y * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int g = blockIdx.x;
  if (r >= d_row) return;
  const float f = *factor;
  const int c0 = g * gs_cols;
  const T* wrow = W + static_cast<size_t>(r) * d_col;
  float mn = INFINITY, mx = -INFINITY;
  for (int c = c0 + lane; c < c0 + gs_cols; c += 32) {
    const float ws = awq_f32<T>(wrow[c]) * (salient[c] != 0.f ? f : 1.f);
    mn = fminf(mn, ws);
    mx = fmaxf(mx, ws);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const AGrid q = awq_grid(mn, mx, maxq, sym);
  if (codes && lane == 0) {
    scales[static_cast<size_t>(g) * d_row + r] = q.s;
    zeros[static_cast<size_t>(g) * d_row + r] = static_cast<uint8_t>(q.z);
  }
  for (int c = c0 + lane; c < c0 + gs_cols; c += 32) {
    const float w = awq_f32<T>(wrow[c]);
    const float tc = salient[c] != 0.f ? f : 1.f;
    const float qz = fminf(fmaxf(rintf(maxq * awq_div(w * tc, q)), -q.z), maxq - q.z);
    if (D_hi) {
      const float dv = w - (q.s * qz) / tc;
      float h, l;
      split_tf32(dv, h, l);
      D_hi[static_cast<size_t>(r) * d_col + c] = h;
      D_lo[static_cast<size_t>(r) * d_col + c] = l;
    }
    if (codes) {
      codes[static_cast<size_t>(r) * d_col + c] = static_cast<uint8_t>(qz + q.z);
      if (r == 0) t_out[c] = tc;
    }
  }
}

// out += sum_i E[i] (D_hi[i] + D_lo[i]), fp64 partials per thread.
__global__ void awq_dot_kernel(const float* __restrict__ E, const float* __restrict__ D_hi,
                               const float* __restrict__ D_lo, size_t n, double* __restrict__ out) {
  double acc = 0.0;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    acc += static_cast<double>(E[i]) * (static_cast<double>(D_hi[i]) + static_cast<double>(D_lo[i]));
#pragma unroll
  for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  __shared__ double red[32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) tot += red[w];
    atomicAdd(out, tot);
  }
}

// The candidate with the smallest error (the earliest on ties).
__global__ void awq_pick_kernel(const double* __restrict__ errors, const float* __restrict__ grid,
                                int n_grid, float* __restrict__ best) {
  int b = 0;
  for (int i = 1; i < n_grid; ++i)
    if (errors[i] < errors[b]) b = i;
  *best = grid[b];
}

__global__ void awq_split_kernel(const float* __restrict__ S, size_t n, float* __restrict__ hi,
                                 float* __restrict__ lo) {
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    float h, l;
    split_tf32(S[i], h, l);
    hi[i] = h;
    lo[i] = l;
  }
}

struct AwqLayout {
  size_t status, salient, grid, errors, best, D_hi, D_lo, S_hi, S_lo, E, total;
};

size_t a256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

AwqLayout awq_layout(int64_t d_row, int64_t d_col, int n_grid) {
  AwqLayout L;
  size_t off = 0;
  L.status = off;
  off += 256;
  L.salient = off;
  off = a256(off + 4 * d_col);
  L.grid = off;
  off = a256(off + 4 * static_cast<size_t>(n_grid));
  L.errors = off;
  off = a256(off + 8 * static_cast<size_t>(n_grid));
  L.best = off;
  off += 256;
  const size_t wd = static_cast<size_t>(d_row) * d_col * 4, ss = static_cast<size_t>(d_col) * d_col * 4;
  L.D_hi = off;
  off = a256(off + wd);
  L.D_lo = off;
  off = a256(off + wd);
  L.S_hi = off;
  off = a256(off + ss);
  L.S_lo = off;
  off = a256(off + ss);
  L.E = off;
  off = a256(off + wd);
  L.total = off;
  return L;
}

template <typename T>
void launch_rtn(const void* W, int d_row, int d_col, int gs_cols, const float* sal, const float* factor,
                float maxq, int sym, float* Dh, float* Dl, uint8_t* codes, float* scales, uint8_t* zeros,
                float* t_out, cudaStream_t st) {
  const int G = d_col / gs_cols;
  dim3 grid(G, (d_row + 7) / 8);
  awq_rtn_kernel<T><<<grid, 256, 0, st>>>(static_cast<const T*>(W), d_row, d_col, gs_cols, sal, factor,
                                          maxq, sym, Dh, Dl, codes, scales, zeros, t_out);
}

}  // namespace

size_t awq_workspace_bytes(int64_t d_row, int64_t d_col, int n_grid) {
  return awq_layout(d_row, d_col, n_grid).total;
}

gptq_status_t launch_awq(const void* W, int w_dtype, int64_t d_row64, int64_t d_col64, const float* S,
                         const double* diag, const gptq_config_t& cfg, float frac, const float* grid_host,
                         int n_grid, uint8_t* codes, float* scales, uint8_t* zeros, float* t_out,
                         double* errors_out, void* ws, cudaStream_t st) {
  const int d_row = static_cast<int>(d_row64), d_col = static_cast<int>(d_col64);
  const AwqLayout L = awq_layout(d_row64, d_col64, n_grid);
  char* base = static_cast<char*>(ws);
  int* status = reinterpret_cast<int*>(base + L.status);
  float* sal = reinterpret_cast<float*>(base + L.salient);
  float* grid = reinterpret_cast<float*>(base + L.grid);
  double* errors = reinterpret_cast<double*>(base + L.errors);
  float* best = reinterpret_cast<float*>(base + L.best);
  float* Dh = reinterpret_cast<float*>(base + L.D_hi);
  float* Dl = reinterpret_cast<float*>(base + L.D_lo);
  float* Sh = reinterpret_cast<float*>(base + L.S_hi);
  float* Sl = reinterpret_cast<float*>(base + L.S_lo);
  float* E = reinterpret_cast<float*>(base + L.E);
  const float maxq = static_cast<float>((1 << cfg.bits) - 1);
  const int gs_cols = cfg.group_size == -1 ? d_col : cfg.group_size;
  const int k = static_cast<int>(std::ceil(static_cast<double>(frac) * d_col - 1e-12));

  GPTQ_CUDA_TRY(cudaMemsetAsync(status, 0, sizeof(int), st));
  GPTQ_CUDA_TRY(cudaMemsetAsync(errors, 0, 8 * static_cast<size_t>(n_grid), st));
  GPTQ_CUDA_TRY(cudaMemcpyAsync(grid, grid_host, 4 * static_cast<size_t>(n_grid), cudaMemcpyHostToDevice, st));
  awq_salient_kernel<<<(d_col + 255) / 256, 256, 0, st>>>(diag, d_col, k, sal);
  GPTQ_LAUNCH_CHECK();
  const size_t nss = static_cast<size_t>(d_col) * d_col, nwd = static_cast<size_t>(d_row) * d_col;
  const int sms = sm_count();
  awq_split_kernel<<<sms * 4, 256, 0, st>>>(S, nss, Sh, Sl);
  GPTQ_LAUNCH_CHECK();
  auto rtn = [&](const float* factor, float* dh, float* dl, uint8_t* c, float* s, uint8_t* z, float* t) {
    if (w_dtype == GPTQ_W_FP32)
      launch_rtn<float>(W, d_row, d_col, gs_cols, sal, factor, maxq, cfg.sym, dh, dl, c, s, z, t, st);
    else if (w_dtype == GPTQ_W_BF16)
      launch_rtn<__nv_bfloat16>(W, d_row, d_col, gs_cols, sal, factor, maxq, cfg.sym, dh, dl, c, s, z, t, st);
    else
      launch_rtn<__half>(W, d_row, d_col, gs_cols, sal, factor, maxq, cfg.sym, dh, dl, c, s, z, t, st);
  };
  for (int i = 0; i < n_grid; ++i) {
    rtn(grid + i, Dh, Dl, nullptr, nullptr, nullptr, nullptr);
    GPTQ_LAUNCH_CHECK();
    TGemmArgs g;
    g.M = d_row;
    g.N = d_col;
    g.K = d_col;
    g.alpha = 1.f;
    g.beta = 0.f;
    g.C = E;
    g.ldc = d_col;
    g.lower = 0;
    g.row_off = 0;
    g.col_off = 0;
    const gptq_status_t s = launch_tgemm_3xtf32(Dh, Dl, d_col, Sh, Sl, d_col, g, status, st);
    if (s != GPTQ_OK) return s;
    awq_dot_kernel<<<sms * 4, 256, 0, st>>>(E, Dh, Dl, nwd, errors + i);
    GPTQ_LAUNCH_CHECK();
  }
  awq_pick_kernel<<<1, 1, 0, st>>>(errors, grid, n_grid, best);
  GPTQ_LAUNCH_CHECK();
  rtn(best, nullptr, nullptr, codes, scales, zeros, t_out);
  GPTQ_LAUNCH_CHECK();
  if (errors_out)
    GPTQ_CUDA_TRY(cudaMemcpyAsync(errors_out, errors, 8 * static_cast<size_t>(n_grid),
                                  cudaMemcpyDeviceToDevice, st));
  return GPTQ_OK;
}

}  // namespace gptq
