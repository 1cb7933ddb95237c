// Step a2: damping, act-order permutation and the inverse Cholesky factor.
//
// [G] GPTQ practical guide (m.lqnn.cn/news/117696):
//   §3.3 damp_percent adds a small term to the Hessian diagonal so that it
//        cannot be singular; desc_act orders the columns;
//   §2.2 columns are put in a fixed order once, by the Hessian diagonal from
//        large to small, and the inverse Hessian is used through a Cholesky
//        factor ("既快又稳定").
//
// What is computed: H = (2/n) S + lambda I with lambda = damp * mean(diag H);
// perm = stable argsort of -diag; Hp = H[perm][:, perm]; U upper triangular
// with Hp^-1 = U^T U.
//
// Route.  With J the index reversal, A = J Hp J = L L^T (ordinary lower
// Cholesky) gives Hp = (J L J)(J L J)^T with J L J upper, so
// U = (J L J)^-1 = J X J with X = L^-1.  X is built together with L in one
// blocked right-looking sweep over 128-column steps k, keeping in the work
// matrix Z
//   * the Schur complement A22 in the trailing lower triangle, and
//   * the running right-hand side Acc = I - L[:, <k] X[<k, :] of L X = I in
//     the lower-left part, where the already-used panels of L used to be.
// Step k:
//   panel kernel   factor the diagonal block, M = L_kk^-1 (every CTA redoes
//                  this small factorization), then in parallel
//                    X_k = [M Acc_k[:, <k], M]   -> U rows (reversed), B rows
//                    P   = A[>k, k] M^T          -> B rows; the panel is zeroed
//                  where B = [X_k^T ; P] (hi/lo TF32 split) is n x 128;
//   update GEMM    Z[>k rows, :] (lower) -= P B^T  on the tensor cores (3xTF32):
//                  the columns left of the diagonal get the Acc update
//                  (-P X_k), the rest the Schur update (-P P^T).
// Cost ~ 2 d^3 / 3 flop, all of it in the tensor-core GEMMs except O(d nb^2).
#include <algorithm>

#include "common.cuh"
#include "tgemm.cuh"

namespace gptq {
namespace {

constexpr int NB = 128;  // step width (K of the update GEMM)

__device__ __forceinline__ unsigned long long ordered_key(double x) {
  unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(x));
  return (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
}

// ---------------------------------------------------------------- stats
__global__ void prep_stats_kernel(const float* __restrict__ S, const double* __restrict__ diag, int d,
                                  double hscale, float damp, unsigned long long* __restrict__ keys,
                                  float* __restrict__ lam_out, int* __restrict__ status) {
  __shared__ double red[32];
  double sum = 0.0;
  int bad = 0;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    const double v = diag ? diag[i] : static_cast<double>(S[static_cast<size_t>(i) * d + i]);
    if (!isfinite(v)) bad = 1;
    sum += v;
    keys[i] = ordered_key(v);
  }
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
  if (bad) atomicOr(status, kStatNonFinite);
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) tot += red[w];
    // mean(diag H) = (2/n) * mean(diag S)
    *lam_out = static_cast<float>(static_cast<double>(damp) * hscale * tot / d);
  }
}

// ---------------------------------------------------------------- order
// rank(i) = #{j : key_j > key_i} + #{j < i : key_j == key_i}; perm[rank] = i.
// Descending diagonal, ties by ascending original index; always a
// permutation (integer keys).
__global__ void prep_rank_kernel(const unsigned long long* __restrict__ keys, int d,
                                 int32_t* __restrict__ perm) {
  __shared__ unsigned long long tile[1024];
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const unsigned long long ki = i < d ? keys[i] : 0ull;
  int rank = 0;
  for (int base = 0; base < d; base += 1024) {
    const int n = min(1024, d - base);
    __syncthreads();
    for (int t = threadIdx.x; t < n; t += blockDim.x) tile[t] = keys[base + t];
    __syncthreads();
    if (i < d) {
#pragma unroll 8
      for (int t = 0; t < n; ++t) {
        const unsigned long long kj = tile[t];
        rank += (kj > ki) | ((kj == ki) & (base + t < i));
      }
    }
  }
  if (i < d) perm[rank] = i;
}

__global__ void iota_kernel(int32_t* __restrict__ perm, int d) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < d) perm[i] = i;
}

// ---------------------------------------------------------------- gather
// Z[i][j] = (2/n) S[q(i)][q(j)] + lambda [i == j] for i >= j, q(i) = perm[d-1-i];
// also U[i][j] = 0 for i > j (the part of U the panel steps do not write).
__global__ void prep_gather_kernel(const float* __restrict__ S, const int32_t* __restrict__ perm, int d,
                                   float hscale, const float* __restrict__ lam,
                                   float* __restrict__ Z, float* __restrict__ U,
                                   int* __restrict__ status) {
  const int bi = blockIdx.y, bj = blockIdx.x;
  if (bj > bi) return;
  const int i = bi * 32 + threadIdx.y * 4;
  const int j = bj * 32 + threadIdx.x;
  const float l = *lam;
  int bad = 0;
  if (j < d) {
    const int qj = perm[d - 1 - j];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int ii = i + r;
      if (ii >= d || j > ii) continue;
      const int qi = perm[d - 1 - ii];
      const int a = max(qi, qj), b = min(qi, qj);
      float v = S[static_cast<size_t>(a) * d + b] * hscale;
      if (ii == j) v += l;
      if (!isfinite(v)) bad = 1;
      Z[static_cast<size_t>(ii) * d + j] = v;
      if (ii > j) U[static_cast<size_t>(ii) * d + j] = 0.f;
    }
  }
  if (bad) atomicOr(status, kStatNonFinite);
}

// ---------------------------------------------------------------- panel step
constexpr int PT = 512;   // threads per panel CTA: thread t owns rows 4(t>>4)..+3,
                          // columns 8(t&15)..+7 of a 128 x 128 block
constexpr int LDM = NB + 4;  // padded row (16-byte aligned rows)

struct PanelArgs {
  float* Z;
  int n;
  int k, b;
  int n_acc;      // CTAs for column slices of X_k left of the diagonal block
  float* Bhi;     // [n][NB]
  float* Blo;
  float* U;       // [n][n] output
  int* status;
};

__device__ __forceinline__ void store_split(float* hi, float* lo, int64_t off, float v) {
  float h, l;
  split_tf32(v, h, l);
  hi[off] = h;
  lo[off] = l;
}

__device__ __forceinline__ void store_split4(float* hi, float* lo, int64_t off, float4 v) {
  float4 h, l;
  split_tf32(v.x, h.x, l.x);
  split_tf32(v.y, h.y, l.y);
  split_tf32(v.z, h.z, l.z);
  split_tf32(v.w, h.w, l.w);
  *reinterpret_cast<float4*>(hi + off) = h;
  *reinterpret_cast<float4*>(lo + off) = l;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}

// Factor the b x b lower block D = Z[k..k+b)^2 and write Mt = (L^-1)^T
// (upper triangular, zeros below) to shared memory.
//
// One right-looking pass over the columns j, on a matrix G held in
// registers (4 x 8 per thread) whose columns < j hold the running
// right-hand side x of L x = I and whose columns >= j hold the Schur
// complement a.  Step j is the rank-1 update of the rows i > j
//   G[i][c] -= (a_ij / a_jj) V[c],   V[c] = x_jc (c < j), a_cj (c > j),
// with G[i][j] set to -a_ij / a_jj (x_ij = 0 - l_ij x_jj, x_jj = 1).  The
// owners of row j and column j publish V (double-buffered) and the pivot
// a_jj; one barrier per column.  At the end L^-1[i][c] = x_ic / sqrt(a_ii).
__device__ bool factor_invert_regs(const float* __restrict__ Z, int64_t ldz, int k, int b,
                                   float* __restrict__ Mt, float* __restrict__ V,
                                   float* __restrict__ piv) {
  const int t = threadIdx.x, rg = t >> 4, cg = t & 15;
  const int r0 = 4 * rg, c0 = 8 * cg;
  const int wmax = ((t >> 5) << 3) + 7;  // last row of this warp
  float g[4][8];
#pragma unroll
  for (int ii = 0; ii < 4; ++ii) {
    const int i = r0 + ii;
    float4 lo4 = make_float4(0.f, 0.f, 0.f, 0.f), hi4 = lo4;
    if (i < b && c0 <= i) {
      const float* src = Z + static_cast<int64_t>(k + i) * ldz + k + c0;
      lo4 = *reinterpret_cast<const float4*>(src);
      if (c0 + 4 <= i) hi4 = *reinterpret_cast<const float4*>(src + 4);
    }
    const float v[8] = {lo4.x, lo4.y, lo4.z, lo4.w, hi4.x, hi4.y, hi4.z, hi4.w};
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) g[ii][cc] = (c0 + cc <= i && i < b) ? v[cc] : 0.f;
  }
  // publish for column j: pivot, row j (c < j) and column j (i > j) into V[j & 1]
  auto publish = [&](int j) {
    float* vb = V + (j & 1) * NB;
    if (rg == (j >> 2)) {
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        if (r0 + ii != j) continue;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const int c = c0 + cc;
          if (c < j) vb[c] = g[ii][cc];
          if (c == j) {
            piv[j] = g[ii][cc];
            g[ii][cc] = 1.f;  // x_jj
          }
        }
      }
    }
    if (cg == (j >> 3)) {
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        if (c0 + cc != j) continue;
#pragma unroll
        for (int ii = 0; ii < 4; ++ii)
          if (r0 + ii > j) vb[r0 + ii] = g[ii][cc];
      }
    }
  };
  publish(0);
  __syncthreads();
  bool notpd = false;
  for (int j = 0; j < b; ++j) {
    const float* vb = V + (j & 1) * NB;
    float ajj = piv[j];
    if (!(ajj > 0.f)) {
      notpd = true;
      ajj = 1.f;
    }
    if (wmax > j) {
      const float inv = 1.f / ajj;
      const float4 va = *reinterpret_cast<const float4*>(vb + c0);
      const float4 vb4 = *reinterpret_cast<const float4*>(vb + c0 + 4);
      const float4 vr = *reinterpret_cast<const float4*>(vb + r0);
      const float vc[8] = {va.x, va.y, va.z, va.w, vb4.x, vb4.y, vb4.z, vb4.w};
      const float rv[4] = {vr.x, vr.y, vr.z, vr.w};
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        if (r0 + ii <= j) continue;
        const float l = rv[ii] * inv;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          g[ii][cc] = (c0 + cc == j) ? -l : fmaf(-l, vc[cc], g[ii][cc]);
      }
    }
    if (j + 1 < b) publish(j + 1);
    __syncthreads();
  }
  // Mt[c][i] = L^-1[i][c] = x_ic / sqrt(a_ii) for c <= i < b, else 0.
#pragma unroll
  for (int ii = 0; ii < 4; ++ii) {
    const int i = r0 + ii;
    const float p = (i < b) ? piv[i] : 1.f;
    const float sc = 1.f / sqrtf(p > 0.f ? p : 1.f);
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      const int c = c0 + cc;
      Mt[c * LDM + i] = (c <= i && i < b) ? g[ii][cc] * sc : 0.f;
    }
  }
  __syncthreads();
  return notpd;
}

__global__ void __launch_bounds__(PT, 1) panel_step_kernel(PanelArgs p) {
  extern __shared__ __align__(16) float sm[];
  float* Mt = sm;                    // [NB][LDM]  (L_kk^-1)^T
  float* T = Mt + NB * LDM;          // [NB][LDM]  role operand tile
  float* V = T + NB * LDM;           // [2][NB]
  float* piv = V + 2 * NB;           // [NB]
  const int n = p.n, k = p.k, b = p.b;
  const int64_t ldz = n;
  const int t = threadIdx.x, rg = t >> 4, cg = t & 15;
  const int r0 = 4 * rg, c0 = 8 * cg;
  const int role = blockIdx.x;

  // Role operand tile, fetched while the diagonal block is factored.
  if (role >= 1) {
    const bool acc = role <= p.n_acc;
    const int base = acc ? (role - 1) * NB : k + b + (role - 1 - p.n_acc) * NB;
    for (int q = t; q < NB * (NB / 4); q += PT) {
      const int rr = q / (NB / 4), c4 = (q % (NB / 4)) * 4;
      const float* src;
      bool ok;
      if (acc) {  // T[q][cc] = Acc[k + q][base + cc]
        ok = rr < b && base + c4 < k;
        src = p.Z + static_cast<int64_t>(k + rr) * ldz + base + c4;
      } else {    // T[rr][q] = A[base + rr][k + q]
        ok = base + rr < n && c4 < b;
        src = p.Z + static_cast<int64_t>(base + rr) * ldz + k + c4;
      }
      cp_async16(T + rr * LDM + c4, ok ? src : p.Z, ok);
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");

  const bool notpd = factor_invert_regs(p.Z, ldz, k, b, Mt, V, piv);
  if (role == 0 && t == 0 && notpd) atomicOr(p.status, kStatNotPD);
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();

  if (role == 0) {
    // X[k + r][k + c] = M[r][c] = Mt[c][r] for c <= r: U[n-1-k-r][n-1-k-c],
    // and B rows k..k+b (B[k + c][r] = Mt[c][r]).
    for (int idx = t; idx < b * b; idx += PT) {
      const int r = idx / b, c = idx % b;
      if (c <= r) p.U[static_cast<int64_t>(n - 1 - k - r) * n + (n - 1 - k - c)] = Mt[c * LDM + r];
    }
    for (int idx = t; idx < b * (NB / 4); idx += PT) {
      const int c = idx / (NB / 4), r4 = (idx % (NB / 4)) * 4;
      store_split4(p.Bhi, p.Blo, static_cast<int64_t>(k + c) * NB + r4,
                   *reinterpret_cast<const float4*>(Mt + c * LDM + r4));
    }
    return;
  }
  float acc[4][8];
#pragma unroll
  for (int ii = 0; ii < 4; ++ii)
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) acc[ii][cc] = 0.f;

  if (role <= p.n_acc) {
    // X_k[r][cbase + cc] = sum_q M[r][q] Acc[q][cc] = sum_q Mt[q][r] T[q][cc]
    const int cbase = (role - 1) * NB;
    const int qmax = min(b, r0 + 4);  // M[r][q] = 0 for q > r
    for (int q = 0; q < qmax; ++q) {
      const float4 m4 = *reinterpret_cast<const float4*>(Mt + q * LDM + r0);
      const float4 t0 = *reinterpret_cast<const float4*>(T + q * LDM + c0);
      const float4 t1 = *reinterpret_cast<const float4*>(T + q * LDM + c0 + 4);
      const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
      const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) acc[ii][cc] = fmaf(mv[ii], tv[cc], acc[ii][cc]);
    }
    const int w = min(NB, k - cbase);
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      const int r = r0 + ii;
      if (r >= b) continue;
      float* urow = p.U + static_cast<int64_t>(n - 1 - (k + r)) * n + (n - 1 - cbase);
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        if (c0 + cc < w) urow[-(c0 + cc)] = acc[ii][cc];
    }
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      if (c0 + cc >= w) continue;
      store_split4(p.Bhi, p.Blo, static_cast<int64_t>(cbase + c0 + cc) * NB + r0,
                   make_float4(acc[0][cc], acc[1][cc], acc[2][cc], acc[3][cc]));
    }
  } else {
    // P[rr][c] = sum_q A[rr][q] M[c][q] = sum_q T[rr][q] Mt[q][c]; zero the panel.
    const int rbase = k + b + (role - 1 - p.n_acc) * NB;
    const int h = min(NB, n - rbase);
    const int qmax = min(b, c0 + 8);  // Mt[q][c] = 0 for q > c
    for (int q = 0; q < qmax; ++q) {
      const float4 m0 = *reinterpret_cast<const float4*>(Mt + q * LDM + c0);
      const float4 m1 = *reinterpret_cast<const float4*>(Mt + q * LDM + c0 + 4);
      const float mv[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
      float av[4];
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) av[ii] = T[(r0 + ii) * LDM + q];
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) acc[ii][cc] = fmaf(av[ii], mv[cc], acc[ii][cc]);
    }
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      const int rr = r0 + ii;
      if (rr >= h) continue;
      const int64_t off = static_cast<int64_t>(rbase + rr) * NB + c0;
      store_split4(p.Bhi, p.Blo, off, make_float4(acc[ii][0], acc[ii][1], acc[ii][2], acc[ii][3]));
      store_split4(p.Bhi, p.Blo, off + 4, make_float4(acc[ii][4], acc[ii][5], acc[ii][6], acc[ii][7]));
    }
    // the panel becomes the (zero) start of the Acc columns of block k
    for (int idx = t; idx < h * (NB / 4); idx += PT) {
      const int rr = idx / (NB / 4), c4 = (idx % (NB / 4)) * 4;
      if (c4 < b)
        *reinterpret_cast<float4*>(p.Z + static_cast<int64_t>(rbase + rr) * ldz + k + c4) =
            make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

}  // namespace

// Workspace layout (byte offsets, each 256-aligned).
struct PrepLayout {
  size_t status, lam, keys, Z, Bhi, Blo, total;
};

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

static PrepLayout prep_layout(int64_t d) {
  PrepLayout L;
  size_t off = 0;
  L.status = off;
  off += 256;
  L.lam = off;
  off += 256;
  L.keys = off;
  off = align256(off + sizeof(unsigned long long) * d);
  L.Z = off;
  off = align256(off + sizeof(float) * d * d);
  L.Bhi = off;
  off = align256(off + sizeof(float) * d * NB);
  L.Blo = off;
  off = align256(off + sizeof(float) * d * NB);
  L.total = off;
  return L;
}

size_t prep_workspace_bytes(int64_t d) { return prep_layout(d).total; }

gptq_status_t launch_prepare(const float* S, const double* diag, int64_t d64, int64_t n_seen,
                             float damp, bool desc_act, float* U, int32_t* perm, void* ws,
                             cudaStream_t st, int* status_host) {
  const int d = static_cast<int>(d64);
  const PrepLayout L = prep_layout(d64);
  char* base = static_cast<char*>(ws);
  int* status = reinterpret_cast<int*>(base + L.status);
  float* lam = reinterpret_cast<float*>(base + L.lam);
  auto* keys = reinterpret_cast<unsigned long long*>(base + L.keys);
  float* Z = reinterpret_cast<float*>(base + L.Z);
  float* Bhi = reinterpret_cast<float*>(base + L.Bhi);
  float* Blo = reinterpret_cast<float*>(base + L.Blo);
  const double hscale = 2.0 / static_cast<double>(n_seen);

  GPTQ_CUDA_TRY(cudaMemsetAsync(status, 0, sizeof(int), st));
  prep_stats_kernel<<<1, 1024, 0, st>>>(S, diag, d, hscale, damp, keys, lam, status);
  GPTQ_LAUNCH_CHECK();
  if (desc_act) {
    prep_rank_kernel<<<(d + 255) / 256, 256, 0, st>>>(keys, d, perm);
  } else {
    iota_kernel<<<(d + 255) / 256, 256, 0, st>>>(perm, d);
  }
  GPTQ_LAUNCH_CHECK();
  {
    dim3 grid((d + 31) / 32, (d + 31) / 32), block(32, 8);
    prep_gather_kernel<<<grid, block, 0, st>>>(S, perm, d, static_cast<float>(hscale), lam, Z, U,
                                                status);
    GPTQ_LAUNCH_CHECK();
  }
  const size_t smem = sizeof(float) * (2 * NB * LDM + 3 * NB);
  GPTQ_CUDA_TRY(cudaFuncSetAttribute(panel_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem)));
  for (int k = 0; k < d; k += NB) {
    const int b = std::min(NB, d - k);
    PanelArgs pa;
    pa.Z = Z;
    pa.n = d;
    pa.k = k;
    pa.b = b;
    pa.n_acc = (k + NB - 1) / NB;
    pa.Bhi = Bhi;
    pa.Blo = Blo;
    pa.U = U;
    pa.status = status;
    const int n_pan = (d - k - b + NB - 1) / NB;
    panel_step_kernel<<<1 + pa.n_acc + n_pan, PT, smem, st>>>(pa);
    GPTQ_LAUNCH_CHECK();
    if (k + b < d) {
      TGemmArgs g;
      g.M = d - k - b;
      g.N = d;
      g.K = NB;
      g.alpha = -1.f;
      g.beta = 1.f;
      g.C = Z + static_cast<int64_t>(k + b) * d;
      g.ldc = d;
      g.lower = 1;
      g.row_off = k + b;
      g.col_off = 0;
      const gptq_status_t s = launch_tgemm_3xtf32(Bhi + static_cast<int64_t>(k + b) * NB,
                                                  Blo + static_cast<int64_t>(k + b) * NB, NB, Bhi, Blo,
                                                  NB, g, st);
      if (s != GPTQ_OK) return s;
    }
  }
  GPTQ_CUDA_TRY(cudaMemcpyAsync(status_host, status, sizeof(int), cudaMemcpyDeviceToHost, st));
  return GPTQ_OK;
}

}  // namespace gptq
