// Steps a3 + a4: the column loop with OBQ error feedback and the 128-column
// lazy batch update.
//
// [G] GPTQ practical guide (m.lqnn.cn/news/117696):
//   §2.1 quantizing one weight is compensated on the weights not yet
//        quantized, in the direction given by the inverse Hessian; through
//        the Cholesky factor U (H^-1 = U^T U) this is
//        w_F -= (w_j - quant(w_j)) / U_jj * U[j, F];
//   §2.2 the columns go in one fixed order and the compensation is batched:
//        quantize 128 columns, then update all remaining columns with one
//        matrix multiply;
//   §3.3 every group_size consecutive columns share one scale and zero point.
// [S] ms-swift review, GPTQ section: sym=True selects a symmetric grid.
//
// Kernels (per layer):
//   load       W (bf16/fp16/fp32) -> fp32 working copy in processing order,
//              g_idx, non-finite check
//   rowparams  group_size = -1 only: one (scale, zero) per row from the
//              initial row
//   per 128-column block [i1, i2):
//     column   row-parallel sequential loop over the block's columns:
//              8 lanes own one row (16 columns each, in registers), the
//              block of U sits in shared memory, the pivot column's value is
//              broadcast with one shuffle per column; group min/max by
//              shuffles; writes codes (original column order), scales,
//              zeros, and Err = the scaled errors of the block
//     trailing W[:, i2:] -= Err U[i1:i2, i2:] on the tensor cores (3xTF32,
//              fp32-accurate), in two levels: inside each 512-column
//              super-block after every block, and for all columns right of
//              the super-block once per super-block with K = 512 (the same
//              sum in another order; a quarter of the read-modify-write
//              traffic on W).  A = Err (hi/lo, written by the column
//              kernel), B = U^T rows (hi/lo, split once per call)
//
// The grid of a group (fp32 working values):
//   asym: xmin = min(0, min w), xmax = max(0, max w), span = xmax - xmin
//   sym:  a = max(-xmin, xmax), span = 2a;  an empty range uses [-1, 1]
//   s = span / maxq (stored), z = rint(-xmin / s) (asym) or (maxq + 1)/2
//   code = clamp(rint(w / s) + z, 0, maxq), round half to even.
// Every quotient w / s is taken as maxq * (w / span), with w / span
// rounded as IEEE division rounds it, so that a weight exactly at a grid
// midpoint (the symmetric grid puts -a at -maxq/2) stays exactly there and
// half-to-even decides it, whatever way the stored scale was rounded.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "tgemm.cuh"

namespace gptq {
namespace {

constexpr int CB = 128;            // block width (blocksize)
constexpr int SB = 4 * CB;         // super-block of the two-level lazy update
// 8 lanes per row, 4 rows per warp: the per-column work that a row's lanes
// all repeat (the grid decision, the error, the look-ahead FMA, the
// shuffles) is shared by fewer lanes than with 16 per row, and a warp's
// instructions serve 4 rows instead of 2; with 4 (8 rows per warp, one warp
// per scheduler) the chain's latency is no longer hidden.  Measured on the
// 4096 x 4096 quantize: 16 lanes 1.334 ms, 8 lanes 1.241 ms, 4 lanes 1.350 ms.
constexpr int LPR = 8;             // lanes per row
constexpr int CPL = CB / LPR;      // columns of a row held by one lane (registers)
constexpr int USEG = CPL + 4;      // padded CPL-column segment of a U row in smem
constexpr int UROW = LPR * USEG;   // padded U row
constexpr int CL_THREADS = 128;    // 4 warps, 16 rows per CTA, 2 CTAs per SM
constexpr int CL_ROWS = CL_THREADS / LPR;

struct QParams {
  float s;     // stored scale, span / maxq
  float span;  // xmax - xmin, or 2a
  float rsp;   // 1 / span (IEEE-rounded)
  float z;     // zero point
};

// x / span as IEEE division rounds it: q0 = x * RN(1/span), then one
// correction by the residual x - span * q0, which a fused multiply-add gives
// exactly.  With a correctly rounded reciprocal this one step yields the
// correctly rounded quotient (Markstein's division theorem); a GPU test
// checks it bit for bit against CUDA's IEEE division.
__device__ __forceinline__ float div_span(float x, const QParams& p) {
  const float q0 = x * p.rsp;
  const float res = fmaf(-q0, p.span, x);
  return fmaf(res, p.rsp, q0);
}

__device__ __forceinline__ QParams grid_from_span(float span, float neg_xmin, float maxq, int sym) {
  QParams p;
  p.span = span;
  p.s = span / maxq;
  p.rsp = 1.f / span;
  p.z = sym ? 0.5f * (maxq + 1.f) : rintf(maxq * div_span(neg_xmin, p));
  return p;
}

__device__ __forceinline__ QParams grid_params(float xmin, float xmax, float maxq, int sym) {
  xmin = fminf(xmin, 0.f);
  xmax = fmaxf(xmax, 0.f);
  if (sym) {
    float a = fmaxf(-xmin, xmax);
    if (a == 0.f) a = 1.f;
    return grid_from_span(2.f * a, a, maxq, 1);
  }
  if (xmin == xmax) {
    xmin = -1.f;
    xmax = 1.f;
  }
  return grid_from_span(xmax - xmin, -xmin, maxq, 0);
}

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
template <>
__device__ __forceinline__ float to_f32<__half>(__half v) {
  return __half2float(v);
}

// Wf[r][i] = W[r][perm[i]]; g_idx[perm[i]] = i / gs.  Each thread takes
// LW_ROWS rows of one column, all loads issued before the stores.
constexpr int LW_ROWS = 8;

template <typename T>
__global__ void load_w_kernel(const T* __restrict__ W, const int32_t* __restrict__ perm, int d_row,
                              int d_col, int gs, float* __restrict__ Wf, int32_t* __restrict__ g_idx,
                              int* __restrict__ status) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= d_col) return;
  const int src = perm[i];
  if (blockIdx.y == 0) g_idx[src] = gs > 0 ? i / gs : 0;
  int bad = 0;
  for (int r0 = blockIdx.y * LW_ROWS; r0 < d_row; r0 += gridDim.y * LW_ROWS) {
    float v[LW_ROWS];
#pragma unroll
    for (int j = 0; j < LW_ROWS; ++j)
      v[j] = r0 + j < d_row ? to_f32<T>(W[static_cast<size_t>(r0 + j) * d_col + src]) : 0.f;
#pragma unroll
    for (int j = 0; j < LW_ROWS; ++j) {
      if (r0 + j >= d_row) break;
      if (!isfinite(v[j])) bad = 1;
      Wf[static_cast<size_t>(r0 + j) * d_col + i] = v[j];
    }
  }
  if (bad) atomicOr(status, kStatNonFinite);
}

// group_size = -1: (scale, zero) per row from the initial row.
__global__ void row_params_kernel(const float* __restrict__ Wf, int d_col, float maxq, int sym,
                                  float* __restrict__ scales, uint8_t* __restrict__ zeros,
                                  float* __restrict__ spans) {
  __shared__ float smn[32], smx[32];
  const int r = blockIdx.x;
  const float* w = Wf + static_cast<size_t>(r) * d_col;
  float mn = INFINITY, mx = -INFINITY;
  for (int i = threadIdx.x; i < d_col; i += blockDim.x) {
    mn = fminf(mn, w[i]);
    mx = fmaxf(mx, w[i]);
  }
  for (int o = 16; o; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if ((threadIdx.x & 31) == 0) {
    smn[threadIdx.x >> 5] = mn;
    smx[threadIdx.x >> 5] = mx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < static_cast<int>(blockDim.x >> 5); ++k) {
      mn = fminf(mn, smn[k]);
      mx = fmaxf(mx, smx[k]);
    }
    const QParams p = grid_params(mn, mx, maxq, sym);
    scales[r] = p.s;
    zeros[r] = static_cast<uint8_t>(p.z);
    spans[r] = p.span;
  }
}

struct ColumnArgs {
  float* Wf;            // [d_row, d_col] working copy (processing order)
  int d_row, d_col;
  int i1, ncols;        // block start and width (multiple of 32, <= CB)
  const float* U;       // [d_col, d_col]
  const int32_t* perm;  // processing position -> original column
  float maxq;
  int gs, sym;
  uint8_t* codes;       // [d_row, d_col] original order
  float* scales;        // [G, d_row]
  uint8_t* zeros;       // [G, d_row]
  float* Err_hi;        // [d_row, SB] scaled errors of the super-block, TF32 split;
  float* Err_lo;        // this block writes columns [err_col0, err_col0 + ncols)
  int err_col0;
  const float* row_span;  // group_size = -1: span of each row's grid
};

__global__ void __launch_bounds__(CL_THREADS, 2) column_block_kernel(ColumnArgs a) {
  extern __shared__ __align__(16) float smem[];
  float* Us = smem;                                  // [CB][UROW]
  float* inv_d = Us + CB * UROW;                     // [CB]
  float* err_s = inv_d + CB;                         // [CL_ROWS][CB + 1]
  uint8_t* code_s = reinterpret_cast<uint8_t*>(err_s + CL_ROWS * (CB + 1));  // [CL_ROWS][CB]

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int row_local = tid / LPR;
  const int sub = lane % LPR;  // this lane holds columns [CPL*sub, CPL*sub + CPL) of the block
  const int r = blockIdx.x * CL_ROWS + row_local;
  const int i1 = a.i1, nc = a.ncols, d = a.d_col;

  // U block, rows/cols [i1, i1 + nc), padded by segment: 16-byte async
  // copies (zero-filled outside the block), all in flight at once.
  for (int q = tid; q < CB * (CB / 4); q += CL_THREADS) {
    const int jj = q / (CB / 4), c4 = (q % (CB / 4)) * 4;
    const bool inb = jj < nc && c4 < nc;
    const float* src = inb ? a.U + static_cast<size_t>(i1 + jj) * d + i1 + c4 : a.U;
    float* dst = Us + jj * UROW + (c4 / CPL) * USEG + (c4 % CPL);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(inb ? 16 : 0)
                 : "memory");
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  for (int jj = tid; jj < CB; jj += CL_THREADS)
    inv_d[jj] = jj < nc ? 1.f / Us[jj * UROW + (jj / CPL) * USEG + (jj % CPL)] : 0.f;
  // U is read-only here: the loads above may overlap the previous kernel
  // (programmatic dependent launch); W, Err, codes and scales may not.
  griddep_wait();
  griddep_launch_dependents();

  float w[CPL];
  const bool row_ok = r < a.d_row;
  const float* wrow = a.Wf + static_cast<size_t>(r) * d + i1 + CPL * sub;
#pragma unroll
  for (int k = 0; k < CPL; k += 4) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row_ok && CPL * sub + k < nc) v = *reinterpret_cast<const float4*>(wrow + k);
    w[k] = v.x;
    w[k + 1] = v.y;
    w[k + 2] = v.z;
    w[k + 3] = v.w;
  }
  QParams p{1.f, 1.f, 1.f, 0.f};
  if (a.gs <= 0 && row_ok) {
    p.s = a.scales[r];
    p.span = a.row_span[r];
    p.rsp = 1.f / p.span;
    p.z = static_cast<float>(a.zeros[r]);
  }
  __syncthreads();

  float e_own[CPL], q_own[CPL];
#pragma unroll
  for (int k = 0; k < CPL; ++k) e_own[k] = q_own[k] = 0.f;
  const int src_base = lane & ~(LPR - 1);
  // Every lane carries the value of the column being quantized (v) and of
  // the next column as it stood before the current column's update (nx):
  // v_{j+1} = nx - e_j U[j][j+1] is one FMA after e_j (the same FMA the
  // owner lane does), so the shuffle that fetches the following nx from
  // its owner runs beside the next decision instead of in front of it.
  float v = __shfl_sync(0xffffffffu, w[0], src_base);
  float nx = __shfl_sync(0xffffffffu, w[1], src_base);
  for (int seg = 0; seg < nc / CPL; ++seg) {
    const int seg_start = i1 + CPL * seg;
    const bool gstart = a.gs > 0 && (seg_start % a.gs) == 0;
    const float* urow_base = Us + (CPL * seg) * UROW + sub * USEG;
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
      if (k == 0 && gstart) {
        // Group [seg_start, seg_start + gs): lanes seg .. seg + gs/CPL - 1 of the row.
        float mn = INFINITY, mx = -INFINITY;
        if (sub >= seg && sub < seg + a.gs / CPL) {
#pragma unroll
          for (int t = 0; t < CPL; ++t) {
            mn = fminf(mn, w[t]);
            mx = fmaxf(mx, w[t]);
          }
        }
#pragma unroll
        for (int o = 1; o < LPR; o <<= 1) {
          mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        p = grid_params(mn, mx, a.maxq, a.sym);
        if (sub == 0 && row_ok) {
          const int g = seg_start / a.gs;
          a.scales[static_cast<size_t>(g) * a.d_row + r] = p.s;
          a.zeros[static_cast<size_t>(g) * a.d_row + r] = static_cast<uint8_t>(p.z);
        }
      }
      const int j = CPL * seg + k;
      // code - z = clamp(rint(v / s), -z, maxq - z); dq = s (code - z)
      const float qz = fminf(fmaxf(rintf(a.maxq * div_span(v, p)), -p.z), a.maxq - p.z);
      const float e = (v - p.s * qz) * inv_d[j];
      const int jn = (j + 1) & (CB - 1);
      const float u_next = Us[j * UROW + (jn / CPL) * USEG + (jn % CPL)];
      v = fmaf(-e, u_next, nx);
      const float* urow = urow_base + k * UROW;
#pragma unroll
      for (int t = 0; t < CPL; t += 4) {
        const float4 u4 = *reinterpret_cast<const float4*>(urow + t);
        w[t] = fmaf(-e, u4.x, w[t]);
        w[t + 1] = fmaf(-e, u4.y, w[t + 1]);
        w[t + 2] = fmaf(-e, u4.z, w[t + 2]);
        w[t + 3] = fmaf(-e, u4.w, w[t + 3]);
      }
      // nx for column j+1: column j+2 after column j's update, from its owner
      nx = __shfl_sync(0xffffffffu, w[(k + 2) % CPL], src_base | ((seg + (k + 2) / CPL) % LPR));
      // The owner lane keeps the error and code of its own columns in
      // registers (no shared-memory stores inside the loop, so the next
      // columns' U loads can be issued early).
      if (sub == seg) {
        e_own[k] = e;
        q_own[k] = qz + p.z;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < CPL; ++k) {
    err_s[row_local * (CB + 1) + CPL * sub + k] = e_own[k];
    code_s[row_local * CB + CPL * sub + k] = static_cast<uint8_t>(q_own[k]);
  }
  __syncthreads();
  // Err block and codes (original column order) for this CTA's rows.
  for (int idx = tid; idx < CL_ROWS * nc; idx += CL_THREADS) {
    const int rl = idx / nc, c = idx % nc;
    const int rr = blockIdx.x * CL_ROWS + rl;
    if (rr >= a.d_row) continue;
    float h, l;
    split_tf32(err_s[rl * (CB + 1) + c], h, l);
    a.Err_hi[static_cast<size_t>(rr) * SB + a.err_col0 + c] = h;
    a.Err_lo[static_cast<size_t>(rr) * SB + a.err_col0 + c] = l;
    a.codes[static_cast<size_t>(rr) * d + a.perm[i1 + c]] = code_s[rl * CB + c];
  }
}

// Ut = U^T split into TF32 hi/lo (32 x 32 tiles through shared memory).
// The trailing updates read Ut[n][k] only for n > k (the columns right of
// a block, against its rows), so the tiles of U below its diagonal block
// (their transposes lie above Ut's diagonal) are skipped.
__global__ void transpose_split_kernel(const float* __restrict__ U, int d, float* __restrict__ Ut_hi,
                                       float* __restrict__ Ut_lo) {
  __shared__ float t[32][33];
  if (blockIdx.x < blockIdx.y) return;
  const int bx = blockIdx.x * 32, by = blockIdx.y * 32;
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int i = by + r, j = bx + threadIdx.x;
    t[r][threadIdx.x] = (i < d && j < d) ? U[static_cast<size_t>(i) * d + j] : 0.f;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int j = bx + r, i = by + threadIdx.x;
    if (i < d && j < d) {
      float h, l;
      split_tf32(t[threadIdx.x][r], h, l);
      Ut_hi[static_cast<size_t>(j) * d + i] = h;
      Ut_lo[static_cast<size_t>(j) * d + i] = l;
    }
  }
}

}  // namespace

constexpr size_t kColumnSmem =
    sizeof(float) * (CB * UROW + CB + CL_ROWS * (CB + 1)) + CL_ROWS * CB;

struct QuantLayout {
  size_t status, row_span, Wf, Err_hi, Err_lo, Ut_hi, Ut_lo, total;
};

static size_t align256q(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

static QuantLayout quant_layout(int64_t d_row, int64_t d_col) {
  QuantLayout L;
  size_t off = 0;
  L.status = off;
  off += 256;
  L.row_span = off;
  off = align256q(off + sizeof(float) * d_row);
  L.Wf = off;
  off = align256q(off + sizeof(float) * d_row * d_col);
  L.Err_hi = off;
  off = align256q(off + sizeof(float) * d_row * SB);
  L.Err_lo = off;
  off = align256q(off + sizeof(float) * d_row * SB);
  L.Ut_hi = off;
  off = align256q(off + sizeof(float) * d_col * d_col);
  L.Ut_lo = off;
  off = align256q(off + sizeof(float) * d_col * d_col);
  L.total = off;
  return L;
}

size_t quant_workspace_bytes(int64_t d_row, int64_t d_col) { return quant_layout(d_row, d_col).total; }

gptq_status_t launch_quantize(const void* W, int w_dtype, int64_t d_row64, int64_t d_col64,
                              const float* U, const int32_t* perm, const gptq_config_t& cfg,
                              uint8_t* codes, float* scales, uint8_t* zeros, int32_t* g_idx,
                              void* ws, cudaStream_t st) {
  const int d_row = static_cast<int>(d_row64), d_col = static_cast<int>(d_col64);
  const QuantLayout L = quant_layout(d_row64, d_col64);
  char* base = static_cast<char*>(ws);
  int* status = reinterpret_cast<int*>(base + L.status);
  float* row_span = reinterpret_cast<float*>(base + L.row_span);
  float* Wf = reinterpret_cast<float*>(base + L.Wf);
  float* Err_hi = reinterpret_cast<float*>(base + L.Err_hi);
  float* Err_lo = reinterpret_cast<float*>(base + L.Err_lo);
  float* Ut_hi = reinterpret_cast<float*>(base + L.Ut_hi);
  float* Ut_lo = reinterpret_cast<float*>(base + L.Ut_lo);
  const float maxq = static_cast<float>((1 << cfg.bits) - 1);
  const int gs = cfg.group_size;

  GPTQ_CUDA_TRY(cudaMemsetAsync(status, 0, sizeof(int), st));
  {
    dim3 grid((d_col + 255) / 256, std::min((d_row + LW_ROWS - 1) / LW_ROWS, 4096));
    if (w_dtype == GPTQ_W_FP32)
      load_w_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(W), perm, d_row, d_col, gs,
                                                 Wf, g_idx, status);
    else if (w_dtype == GPTQ_W_BF16)
      load_w_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(W), perm,
                                                         d_row, d_col, gs, Wf, g_idx, status);
    else
      load_w_kernel<__half><<<grid, 256, 0, st>>>(static_cast<const __half*>(W), perm, d_row, d_col,
                                                  gs, Wf, g_idx, status);
    GPTQ_LAUNCH_CHECK();
  }
  if (gs <= 0) {
    row_params_kernel<<<d_row, 256, 0, st>>>(Wf, d_col, maxq, cfg.sym, scales, zeros, row_span);
    GPTQ_LAUNCH_CHECK();
  }
  {
    dim3 grid((d_col + 31) / 32, (d_col + 31) / 32), block(32, 8);
    transpose_split_kernel<<<grid, block, 0, st>>>(U, d_col, Ut_hi, Ut_lo);
    GPTQ_LAUNCH_CHECK();
  }
  GPTQ_CUDA_TRY(cudaFuncSetAttribute(column_block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kColumnSmem)));
  // Two CTAs per SM need the largest shared-memory carveout.
  GPTQ_CUDA_TRY(cudaFuncSetAttribute(column_block_kernel,
                                     cudaFuncAttributePreferredSharedMemoryCarveout, 100));
  // Two-level lazy update: after each 128-column block only the rest of its
  // 512-column super-block is updated; after the super-block, everything to
  // its right is updated in one K = 512 product.  The sum is the same as the
  // single-level schedule up to the order of fp32 additions.
  auto trailing = [&](int k0, int k_len, int e0, int n0, int n1) -> gptq_status_t {
    TGemmArgs g;
    g.M = d_row;
    g.N = n1 - n0;
    g.K = k_len;
    g.alpha = -1.f;
    g.beta = 1.f;
    g.C = Wf + n0;
    g.ldc = d_col;
    g.lower = 0;
    g.row_off = 0;
    g.col_off = 0;
    return launch_tgemm_3xtf32(Err_hi + e0, Err_lo + e0, SB,
                               Ut_hi + static_cast<int64_t>(n0) * d_col + k0,
                               Ut_lo + static_cast<int64_t>(n0) * d_col + k0, d_col, g, status, st);
  };
  for (int sb0 = 0; sb0 < d_col; sb0 += SB) {
    const int sb1 = std::min(sb0 + SB, d_col);
    for (int i1 = sb0; i1 < sb1; i1 += CB) {
      const int nc = std::min(CB, sb1 - i1);
      ColumnArgs ca;
      ca.Wf = Wf;
      ca.d_row = d_row;
      ca.d_col = d_col;
      ca.i1 = i1;
      ca.ncols = nc;
      ca.U = U;
      ca.perm = perm;
      ca.maxq = maxq;
      ca.gs = gs;
      ca.sym = cfg.sym;
      ca.codes = codes;
      ca.scales = scales;
      ca.zeros = zeros;
      ca.Err_hi = Err_hi;
      ca.Err_lo = Err_lo;
      ca.err_col0 = i1 - sb0;
      ca.row_span = row_span;
      GPTQ_CUDA_TRY(launch_pdl(column_block_kernel, dim3((d_row + CL_ROWS - 1) / CL_ROWS),
                               dim3(CL_THREADS), kColumnSmem, st, ca));
      GPTQ_LAUNCH_CHECK();
      const int i2 = i1 + nc;
      if (i2 < sb1) {
        const gptq_status_t s = trailing(i1, nc, i1 - sb0, i2, sb1);
        if (s != GPTQ_OK) return s;
      }
    }
    if (sb1 < d_col) {
      const gptq_status_t s = trailing(sb0, sb1 - sb0, 0, sb1, d_col);
      if (s != GPTQ_OK) return s;
    }
  }
  return GPTQ_OK;
}

}  // namespace gptq

namespace {
__global__ void div_span_probe_kernel(const float* __restrict__ x, const float* __restrict__ span,
                                      int n, float* __restrict__ q_grid,
                                      float* __restrict__ q_ieee) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  gptq::QParams p;
  p.span = span[i];
  p.rsp = 1.f / p.span;
  q_grid[i] = gptq::div_span(x[i], p);
  q_ieee[i] = __fdiv_rn(x[i], span[i]);
}
}  // namespace

// Test hook (not part of the public header): the grid's quotient x / span
// next to CUDA's IEEE division of the same operands, for n pairs.
extern "C" GPTQ_API int gptq_internal_div_span(const float* x, const float* span, int n,
                                               float* q_grid, float* q_ieee, gptq_stream_t stream) {
  if (n <= 0) return GPTQ_OK;
  div_span_probe_kernel<<<(n + 255) / 256, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      x, span, n, q_grid, q_ieee);
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}
