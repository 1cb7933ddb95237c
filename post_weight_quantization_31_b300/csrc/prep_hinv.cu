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
// Route: with J the index reversal, A = J Hp J = L L^T (ordinary lower
// Cholesky) gives Hp = (J L J)(J L J)^T with J L J upper, hence
// U = (J L J)^-1 = J L^-1 J.  So the kernels run a standard blocked lower
// Cholesky and a blocked lower-triangular inverse on A = J Hp J, and the
// last kernel reverses indices while writing U.  Cost ~ 2 d^3 / 3 flop.
//
//   1. stats   mean of diag H (fp64 sum), lambda, ordered sort keys
//   2. order   perm by rank counting (stable, exact on integer keys)
//   3. gather  A[i][j] = (2/n) S[q(i)][q(j)] + lambda [i==j], q(i) = perm[d-1-i]
//   4. blocked Cholesky with nb = 128:
//        diagonal block: factor and invert in one pass (shared memory); the
//          inverse of the diagonal block overwrites it;
//        panel:  A21 <- A21 L11^-T           (GEMM with the block inverse)
//        update: A22 <- A22 - A21 A21^T      (lower tiles only)
//   5. blocked triangular inverse, bottom-up over power-of-two levels:
//        X21 = -X22 (A21 X11)   for every pair of adjacent diagonal blocks
//   6. U[i][j] = X[d-1-i][d-1-j] for i <= j, 0 below the diagonal.
#include <algorithm>

#include "common.cuh"
#include "sgemm.cuh"

namespace gptq {
namespace {

constexpr int NB = 128;  // Cholesky block

__device__ __forceinline__ unsigned long long ordered_key(double x) {
  unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(x));
  return (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
}

// ---------------------------------------------------------------- 1. stats
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

// ---------------------------------------------------------------- 2. order
// rank(i) = #{j : key_j > key_i} + #{j < i : key_j == key_i}; perm[rank] = i.
// Descending diagonal, ties by ascending original index.
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

// ---------------------------------------------------------------- 3. gather
__global__ void prep_gather_kernel(const float* __restrict__ S, const int32_t* __restrict__ perm, int d,
                                   float hscale, const float* __restrict__ lam,
                                   float* __restrict__ A, int* __restrict__ status) {
  // 32 x 32 tiles of the lower triangle of A.
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
      A[static_cast<size_t>(ii) * d + j] = v;
    }
  }
  if (bad) atomicOr(status, kStatNonFinite);
}

// ---------------------------------------------------------------- 4a. diagonal block
// Factor the b x b lower block at (k0, k0) (b <= NB) and replace it by the
// inverse of its Cholesky factor (zeros above the diagonal).  One pass over
// j: with a the running Schur complement and x the running right-hand side
// of L x = I,
//   step j:  a[i][k] -= a[i][j] a[k][j] / a[j][j]      (j < k <= i)
//            x[i][c] -= a[i][j] x[j][c] / a[j][j]      (i > j, c <= j)
// and finally L^-1[i][c] = x[i][c] / sqrt(a[i][i]).
constexpr int CB_THREADS = 1024;
constexpr int CB_LD = NB + 1;

__global__ void __launch_bounds__(CB_THREADS)
    chol_block_kernel(float* __restrict__ A, int64_t lda, int k0, int b, int* __restrict__ status) {
  extern __shared__ float sm[];
  float* a = sm;                  // [NB][CB_LD]
  float* x = sm + NB * CB_LD;     // [NB][CB_LD]
  float* A0 = A + k0 * lda + k0;
  for (int idx = threadIdx.x; idx < b * b; idx += blockDim.x) {
    const int i = idx / b, k = idx % b;
    a[i * CB_LD + k] = (k <= i) ? A0[i * lda + k] : 0.f;
    x[i * CB_LD + k] = (i == k) ? 1.f : 0.f;
  }
  __syncthreads();
  const int tr = threadIdx.x >> 5;  // rows tr, tr+32, ...
  const int tc = threadIdx.x & 31;  // cols tc, tc+32, ...
  bool notpd = false;
  for (int j = 0; j < b; ++j) {
    float djj = a[j * CB_LD + j];
    if (!(djj > 0.f)) {
      notpd = true;
      djj = 1.f;
    }
    const float inv = 1.f / djj;
    for (int i = tr; i < b; i += 32) {
      if (i <= j) continue;
      const float aij = a[i * CB_LD + j] * inv;
      for (int c = tc; c <= i; c += 32) {
        if (c > j)
          a[i * CB_LD + c] = fmaf(-aij, a[c * CB_LD + j], a[i * CB_LD + c]);
        else
          x[i * CB_LD + c] = fmaf(-aij, x[j * CB_LD + c], x[i * CB_LD + c]);
      }
    }
    __syncthreads();
  }
  if (notpd && threadIdx.x == 0) atomicOr(status, kStatNotPD);
  for (int idx = threadIdx.x; idx < b * b; idx += blockDim.x) {
    const int i = idx / b, c = idx % b;
    float v = 0.f;
    if (c <= i) {
      const float p = a[i * CB_LD + i];
      v = x[i * CB_LD + c] / sqrtf(p > 0.f ? p : 1.f);
    }
    A0[i * lda + c] = v;
  }
}

// ---------------------------------------------------------------- 4b/4c. panel and update
__global__ void __launch_bounds__(GEMM_THREADS) panel_kernel(GemmArgs g) {
  __shared__ GemmSmem s;
  gemm_tile</*B_NK*/ true, false, false>(g, blockIdx.y * GM, blockIdx.x * GN, s);
}

__global__ void __launch_bounds__(GEMM_THREADS) syrk_update_kernel(GemmArgs g) {
  __shared__ GemmSmem s;
  const int m0 = blockIdx.y * GM, n0 = blockIdx.x * GN;
  if (n0 > m0 + GM - 1) return;  // tile entirely above the diagonal
  gemm_tile</*B_NK*/ true, false, false>(g, m0, n0, s);
}

// ---------------------------------------------------------------- 5. triangular inverse
// Level with block size sz: pair p covers X11 = [a, a+sz), X22 = [a+sz, a+sz+s2).
struct TrtriLevel {
  float* A;
  int64_t lda;
  int d, sz;
  float* T;  // workspace, pair p at T + p * sz * sz, leading dimension sz
};

__global__ void __launch_bounds__(GEMM_THREADS) trtri_step1_kernel(TrtriLevel L) {
  // T = A21 * X11  (X11 lower triangular)
  __shared__ GemmSmem s;
  const int p = blockIdx.z;
  const int a = 2 * L.sz * p;
  const int s2 = min(L.sz, L.d - a - L.sz);
  if (s2 <= 0) return;
  GemmArgs g;
  g.M = s2;
  g.N = L.sz;
  g.K = L.sz;
  g.alpha = 1.f;
  g.beta = 0.f;
  g.A = L.A + static_cast<int64_t>(a + L.sz) * L.lda + a;
  g.lda = L.lda;
  g.B = L.A + static_cast<int64_t>(a) * L.lda + a;
  g.ldb = L.lda;
  g.C = L.T + static_cast<int64_t>(p) * L.sz * L.sz;
  g.ldc = L.sz;
  gemm_tile<false, false, /*B_LOWER*/ true>(g, blockIdx.y * GM, blockIdx.x * GN, s);
}

__global__ void __launch_bounds__(GEMM_THREADS) trtri_step2_kernel(TrtriLevel L) {
  // X21 = -X22 * T  (X22 lower triangular), written over A21
  __shared__ GemmSmem s;
  const int p = blockIdx.z;
  const int a = 2 * L.sz * p;
  const int s2 = min(L.sz, L.d - a - L.sz);
  if (s2 <= 0) return;
  GemmArgs g;
  g.M = s2;
  g.N = L.sz;
  g.K = s2;
  g.alpha = -1.f;
  g.beta = 0.f;
  g.A = L.A + static_cast<int64_t>(a + L.sz) * L.lda + a + L.sz;
  g.lda = L.lda;
  g.B = L.T + static_cast<int64_t>(p) * L.sz * L.sz;
  g.ldb = L.sz;
  g.C = L.A + static_cast<int64_t>(a + L.sz) * L.lda + a;
  g.ldc = L.lda;
  gemm_tile<false, /*A_LOWER*/ true, false>(g, blockIdx.y * GM, blockIdx.x * GN, s);
}

// ---------------------------------------------------------------- 6. output
__global__ void prep_output_kernel(const float* __restrict__ X, int d, float* __restrict__ U) {
  const int i = blockIdx.y;
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < d; j += gridDim.x * blockDim.x) {
    float v = 0.f;
    if (j >= i) v = X[static_cast<size_t>(d - 1 - i) * d + (d - 1 - j)];
    U[static_cast<size_t>(i) * d + j] = v;
  }
}

}  // namespace

// Workspace layout (byte offsets, each 256-aligned).
struct PrepLayout {
  size_t status, lam, keys, A, T, total;
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
  L.A = off;
  off = align256(off + sizeof(float) * d * d);
  L.T = off;
  off = align256(off + sizeof(float) * ((d * d) / 4 + NB * NB));
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
  float* A = reinterpret_cast<float*>(base + L.A);
  float* T = reinterpret_cast<float*>(base + L.T);
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
    prep_gather_kernel<<<grid, block, 0, st>>>(S, perm, d, static_cast<float>(hscale), lam, A, status);
    GPTQ_LAUNCH_CHECK();
  }
  // 4. blocked Cholesky
  const size_t cb_smem = sizeof(float) * 2 * NB * CB_LD;
  GPTQ_CUDA_TRY(cudaFuncSetAttribute(chol_block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(cb_smem)));
  for (int k0 = 0; k0 < d; k0 += NB) {
    const int b = std::min(NB, d - k0);
    chol_block_kernel<<<1, CB_THREADS, cb_smem, st>>>(A, d, k0, b, status);
    GPTQ_LAUNCH_CHECK();
    const int rest = d - k0 - b;
    if (rest <= 0) break;
    GemmArgs g;
    g.M = rest;
    g.N = b;
    g.K = b;
    g.alpha = 1.f;
    g.beta = 0.f;
    g.A = A + static_cast<int64_t>(k0 + b) * d + k0;  // panel, in place
    g.lda = d;
    g.B = A + static_cast<int64_t>(k0) * d + k0;  // block inverse, used as [N, K]
    g.ldb = d;
    g.C = A + static_cast<int64_t>(k0 + b) * d + k0;
    g.ldc = d;
    panel_kernel<<<dim3(1, (rest + GM - 1) / GM), GEMM_THREADS, 0, st>>>(g);
    GPTQ_LAUNCH_CHECK();
    GemmArgs u;
    u.M = rest;
    u.N = rest;
    u.K = b;
    u.alpha = -1.f;
    u.beta = 1.f;
    u.A = A + static_cast<int64_t>(k0 + b) * d + k0;
    u.lda = d;
    u.B = u.A;
    u.ldb = d;
    u.C = A + static_cast<int64_t>(k0 + b) * d + (k0 + b);
    u.ldc = d;
    syrk_update_kernel<<<dim3((rest + GN - 1) / GN, (rest + GM - 1) / GM), GEMM_THREADS, 0, st>>>(u);
    GPTQ_LAUNCH_CHECK();
  }
  // 5. triangular inverse (diagonal blocks already inverted)
  for (int sz = NB; sz < d; sz *= 2) {
    TrtriLevel lv{A, d, d, sz, T};
    const int pairs = (d + 2 * sz - 1) / (2 * sz);
    dim3 grid((sz + GN - 1) / GN, (sz + GM - 1) / GM, pairs);
    trtri_step1_kernel<<<grid, GEMM_THREADS, 0, st>>>(lv);
    GPTQ_LAUNCH_CHECK();
    trtri_step2_kernel<<<grid, GEMM_THREADS, 0, st>>>(lv);
    GPTQ_LAUNCH_CHECK();
  }
  // 6. reversed copy into U
  prep_output_kernel<<<dim3((d + 255) / 256, d), 256, 0, st>>>(A, d, U);
  GPTQ_LAUNCH_CHECK();
  GPTQ_CUDA_TRY(cudaMemcpyAsync(status_host, status, sizeof(int), cudaMemcpyDeviceToHost, st));
  return GPTQ_OK;
}

}  // namespace gptq
