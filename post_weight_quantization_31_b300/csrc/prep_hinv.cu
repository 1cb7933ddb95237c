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
//   factor kernel  factor the diagonal block, M = L_kk^-1 (one CTA);
//   role kernel    in parallel
//                    X_k = [M Acc_k[:, <k], M]   -> U rows (reversed), B rows
//                    P   = A[>k, k] M^T          -> B rows; the panel is zeroed
//                  where B = [X_k^T ; P] (hi/lo TF32 split) is n x 128;
//   update GEMM    Z[>k rows, :] (lower) -= P B^T  on the tensor cores (3xTF32):
//                  the columns left of the diagonal get the Acc update
//                  (-P X_k), the rest the Schur update (-P P^T); first the
//                  tiles step k + 1 reads, then the rest, beside the factor
//                  kernel of step k + 1 (see launch_prepare).
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
// The sort keys of the diagonal, and per block of 256 entries the fp64 sum
// of the diagonal (`part`, summed in a fixed order by prep_diag_kernel, so
// that lambda does not depend on the schedule).  Also perm = identity when
// there is no act-order.
constexpr int ST_THREADS = 256;

__global__ void prep_stats_kernel(const float* __restrict__ S, const double* __restrict__ diag, int d,
                                  unsigned long long* __restrict__ keys, double* __restrict__ part,
                                  int32_t* __restrict__ iota_perm, int* __restrict__ status) {
  __shared__ double red[ST_THREADS / 32];
  const int i = blockIdx.x * ST_THREADS + threadIdx.x;
  double v = 0.0;
  if (i < d) {
    v = diag ? diag[i] : static_cast<double>(S[static_cast<size_t>(i) * d + i]);
    if (!isfinite(v)) atomicOr(status, kStatNonFinite);
    keys[i] = ordered_key(v);
    if (iota_perm) iota_perm[i] = i;
  }
  double sum = v;
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int w = 0; w < ST_THREADS / 32; ++w) tot += red[w];
    part[blockIdx.x] = tot;
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

// ---------------------------------------------------------------- gather
// prep_diag_kernel: Z[i][i] + zlo[i] = (2/n) S_ii + lambda, formed in fp64 and
// carried as an fp32 pair (see the update GEMM), S_ii taken from the fp64
// diagonal when it is given: the tensor-core sums of S are biased low on the
// diagonal, where every term is positive (about 5e-6 relative per
// 1024-token accumulator fill), and that bias alone moves U by about 1e-6 at
// d_col = 13824.
// prep_gather_kernel: Z[i][j] = (2/n) S[q(i)][q(j)] for i > j, with
// q(i) = perm[d-1-i]; also U[i][j] = 0 for i > j (the part of U the panel
// steps do not write).
__global__ void prep_diag_kernel(const float* __restrict__ S, const double* __restrict__ diag,
                                 const int32_t* __restrict__ perm, int d, double hscale_d, float damp,
                                 const double* __restrict__ part, int nparts, float* __restrict__ Z,
                                 float* __restrict__ zlo, int* __restrict__ status) {
  // lambda = damp * mean(diag H) = damp * (2/n) * mean(diag S), the block sums
  // added in block order.
  double tot = 0.0;
  for (int b = 0; b < nparts; ++b) tot += part[b];
  const float lam = static_cast<float>(static_cast<double>(damp) * hscale_d * tot / d);
  // The diagonal is carried as Z + zlo (see the update GEMM).
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= d) return;
  const int qi = perm[d - 1 - i];
  const double s = diag ? diag[qi] : static_cast<double>(S[static_cast<size_t>(qi) * d + qi]);
  const double v64 = s * hscale_d + static_cast<double>(lam);
  const float v = static_cast<float>(v64);
  Z[static_cast<size_t>(i) * d + i] = v;
  zlo[i] = static_cast<float>(v64 - static_cast<double>(v));
  if (!isfinite(v)) atomicOr(status, kStatNonFinite);
}

// One 32 x 32 tile of Z (rows ii, columns j, lower part) per block of
// 32 x 8 threads, through shared memory: in processing order without
// act-order the entries S[q(j)][q(ii)] of a tile form a block of S whose
// rows are contiguous along ii, so the loads run with the lanes along ii and
// the stores of Z and U with the lanes along j.
__global__ void prep_gather_kernel(const float* __restrict__ S, const int32_t* __restrict__ perm, int d,
                                   float hscale, float* __restrict__ Z, float* __restrict__ U,
                                   int* __restrict__ status) {
  __shared__ float t[32][33];
  const int bi = blockIdx.y, bj = blockIdx.x;
  if (bj > bi) return;
  const int i0 = bi * 32, j0 = bj * 32;
  const int tx = threadIdx.x;
  int bad = 0;
  {  // t[jj][iix] = (2/n) S[max(q(ii), q(j))][min(q(ii), q(j))], ii = i0 + tx
    const int ii = i0 + tx;
    const int qi = ii < d ? perm[d - 1 - ii] : 0;
    for (int jj = threadIdx.y; jj < 32; jj += blockDim.y) {
      const int j = j0 + jj;
      float v = 0.f;
      if (ii < d && j < ii) {
        const int qj = perm[d - 1 - j];
        const int a = max(qi, qj), b = min(qi, qj);
        v = S[static_cast<size_t>(a) * d + b] * hscale;
        if (!isfinite(v)) bad = 1;
      }
      t[jj][tx] = v;
    }
  }
  __syncthreads();
  {  // Z[ii][j] and U[ii][j] = 0 for ii > j, lanes along j (the diagonal: prep_diag_kernel)
    const int j = j0 + tx;
    for (int r = threadIdx.y; r < 32; r += blockDim.y) {
      const int ii = i0 + r;
      if (ii >= d || j >= ii) continue;
      Z[static_cast<size_t>(ii) * d + j] = t[tx][r];
      U[static_cast<size_t>(ii) * d + j] = 0.f;
    }
  }
  if (bad) atomicOr(status, kStatNonFinite);
}

// ---------------------------------------------------------------- panel step
constexpr int PT = 512;   // threads per role CTA
// Threads of the factor CTA: its widest phases (the update of the diagonal
// block after the first sub-panel, and the inverse's block-row sums after
// the last) take 384 threads, and with 384 the factorization's registers
// (up to 168 a thread) hold its 32-entry rows without spilling.
constexpr int FT = 384;
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
  const float* zlo;  // [n] low parts of the diagonal of Z
  int split;         // CTAs per role tile (1, 2 or 4)
  float* Mg;         // [NB][NB] (L_kk^-1)^T, from the factor kernel to the role kernel
  int wait_first;    // factor kernel: wait for the previous kernel before starting
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

// Factor the b x b lower block D = Z[k..k+b)^2 (b a multiple of 32, at most
// NB) and write Mt = (L^-1)^T (Mt[c][i] = L^-1[i][c]) to shared memory,
// which the caller has zeroed (so that Mt is zero above the diagonal of
// L^-1 and outside b).
//
// Blocked over 32-wide sub-panels s, so that the column-by-column chain of
// the factorization runs inside one warp and block barriers are needed only
// between the sub-panel phases:
//   F  one warp factors the 32 x 32 diagonal sub-block in registers (lane i
//      holds row i; each column's entries are broadcast through shared
//      memory);
//   T  the rows below, one thread per row, solve x L_ss^T = d by forward
//      substitution (L_ts = D_ts L_ss^-T);
//   U  the trailing sub-blocks of the diagonal block get D_tu -= L_ts L_us^T.
// L^-1 = M is built by block rows as soon as each row of L is known: in T,
// one more warp inverts the diagonal sub-block (M_ss, back substitution per
// row, no cross-lane traffic); in U, the warps the update leaves idle form
// the sums R_u = sum_{v=u}^{s-1} L_sv M_vu for u < s; in the next F, the
// warps beside the factoring one finish M_su = -M_ss R_u.  So the inverse
// costs one phase after the last sub-panel instead of phases of its own.
// Returns true (in thread 0) if a pivot was not positive.
constexpr int TMLD = 36;  // row stride of the 32 x 32 level products

constexpr int LST = 36;  // row stride of the transposed 32 x 32 diagonal sub-block

// Inverse of the diagonal sub-block s by one warp: lane i computes row i of
// M_ss (back substitution), written transposed into Mt.
__device__ __forceinline__ void invert_diag_block(int s, const float* __restrict__ Ls,
                                                  const float* __restrict__ rdiag,
                                                  float* __restrict__ Mt, int lane) {
  const int w0 = 32 * s;
  float acc[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) acc[c] = (c == lane) ? 1.f : 0.f;
#pragma unroll
  for (int m = 31; m >= 0; --m) {
    const float ym = (m <= lane) ? acc[m] * rdiag[w0 + m] : 0.f;
    Mt[(w0 + m) * LDM + w0 + lane] = ym;
#pragma unroll
    for (int c = 0; c < m; ++c) acc[c] = fmaf(-ym, Ls[(w0 + m) * LDM + w0 + c], acc[c]);
  }
}

// First half of block (tb, sb) of M, sb < tb, by 64 threads (g in [0, 64):
// rows i and i + 16 of the block with i = g % 16, columns 8 (g / 16) .. + 8):
// R[i][c] = sum_{u=sb}^{tb-1} L_{tb,u} M_{u,sb}, into Tm slot sb.  Two rows
// a thread, so that each column value read from shared memory feeds two
// rows; every output is summed in the same order as with one row a thread.
__device__ __forceinline__ void inverse_rows_sum(int tb, int sb, int g, const float* __restrict__ Ls,
                                                 const float* __restrict__ Mt, float* __restrict__ Tm) {
  const int i = g & 15, cg8 = (g >> 4) * 8;
  float acc[2][8];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) acc[h][cc] = 0.f;
  for (int u = sb; u < tb; ++u) {
    const float* li = Ls + (32 * tb + i) * LDM + 32 * u;
#pragma unroll 2
    for (int m = 0; m < 32; m += 4) {
      const float4 x0 = *reinterpret_cast<const float4*>(li + m);
      const float4 x1 = *reinterpret_cast<const float4*>(li + 16 * LDM + m);
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const float4 y = *reinterpret_cast<const float4*>(Mt + (32 * sb + cg8 + cc) * LDM + 32 * u + m);
        acc[0][cc] = fmaf(x0.x, y.x, fmaf(x0.y, y.y, fmaf(x0.z, y.z, fmaf(x0.w, y.w, acc[0][cc]))));
        acc[1][cc] = fmaf(x1.x, y.x, fmaf(x1.y, y.y, fmaf(x1.z, y.z, fmaf(x1.w, y.w, acc[1][cc]))));
      }
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float* tm = Tm + (sb * 32 + i + 16 * h) * TMLD + cg8;
    *reinterpret_cast<float4*>(tm) = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
    *reinterpret_cast<float4*>(tm + 4) = make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
  }
}

// Second half, by 128 threads per sb (g in [0, 128): row i = g % 32,
// columns 8 (g / 32) .. + 8): M_{tb,sb} = -M_{tb,tb} R.
__device__ __forceinline__ void inverse_rows_finish(int tb, int sb, int g, const float* __restrict__ Tm,
                                                    float* __restrict__ Mt) {
  const int i = g & 31, cg8 = (g >> 5) * 8;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int m = 0; m < 32; ++m) {
    const float mv = Mt[(32 * tb + m) * LDM + 32 * tb + i];
    const float4 y0 = *reinterpret_cast<const float4*>(Tm + (sb * 32 + m) * TMLD + cg8);
    const float4 y1 = *reinterpret_cast<const float4*>(Tm + (sb * 32 + m) * TMLD + cg8 + 4);
    acc[0] = fmaf(mv, y0.x, acc[0]);
    acc[1] = fmaf(mv, y0.y, acc[1]);
    acc[2] = fmaf(mv, y0.z, acc[2]);
    acc[3] = fmaf(mv, y0.w, acc[3]);
    acc[4] = fmaf(mv, y1.x, acc[4]);
    acc[5] = fmaf(mv, y1.y, acc[5]);
    acc[6] = fmaf(mv, y1.z, acc[6]);
    acc[7] = fmaf(mv, y1.w, acc[7]);
  }
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) Mt[(32 * sb + cg8 + cc) * LDM + 32 * tb + i] = -acc[cc];
}

__device__ bool factor_invert_blocked(const float* __restrict__ Z, const float* __restrict__ zlo,
                                      int64_t ldz, int k, int b,
                                      float* __restrict__ Mt, float* __restrict__ Ls,
                                      float* __restrict__ rdiag, float* __restrict__ Tm,
                                      float* __restrict__ LT, float* __restrict__ colbuf,
                                      float* __restrict__ LssT) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int nsub = b >> 5;
  // The lower 4-wide chunks of the block (zero elsewhere), all copies in
  // flight at once; then the diagonal gets its low part, hi + lo.
  for (int q = t; q < NB * (NB / 4); q += FT) {
    const int i = q / (NB / 4), c4 = (q % (NB / 4)) * 4;
    const bool ok = i < b && c4 <= i;
    cp_async16(Ls + i * LDM + c4, ok ? Z + static_cast<int64_t>(k + i) * ldz + k + c4 : Z, ok);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  if (t < b) Ls[t * LDM + t] += __ldcg(zlo + k + t);
  __syncthreads();
  bool bad = false;
  for (int s = 0; s < nsub; ++s) {
    const int c0 = 32 * s;
    // block row s - 1 of M, second half, beside the factorization, on the
    // warps that do not share a scheduler with the factoring warp 0
    // (warp w goes to scheduler w mod 4): warps 1-3, 5-7, 9-11 in order.
    const int gf = 32 * (warp - warp / 4 - 1) + lane;
    if ((warp & 3) != 0 && s >= 2 && gf < (s - 1) * 128)
      inverse_rows_finish(s - 1, gf >> 7, gf & 127, Tm, Mt);
    if (warp == 0) {
      // ---- F: Cholesky of the diagonal sub-block, lane = row
      float a[32];
      float* row = Ls + (c0 + lane) * LDM + c0;
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 v = *reinterpret_cast<const float4*>(row + c);
        a[c] = v.x;
        a[c + 1] = v.y;
        a[c + 2] = v.z;
        a[c + 3] = v.w;
      }
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (c > lane) a[c] = 0.f;
      float my_r = 1.f;
      float mypiv = 1.f;  // this lane's pivot (checked after the loop)
      float pn = a[0];  // lane j's current diagonal when column j starts
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float ajj = __shfl_sync(0xffffffffu, pn, j);
        // A pivot that is not positive is replaced by 1 and reported below;
        // no branch in the loop (a branch here made the loop spill).
        if (lane == j) mypiv = ajj;
        ajj = ajj > 0.f ? ajj : 1.f;
        const float r = rsqrtf(ajj);  // 1 / l_jj
        if (lane == j) my_r = r;
        const float l = (lane == j) ? ajj * r : a[j] * r;  // l_ij for lanes i >= j
        a[j] = (lane >= j) ? l : 0.f;
        // Lane j+1's next pivot is its own a[j+1] - l^2: formed here, it does
        // not wait for the broadcast below (the same fma the update does).
        if (j + 1 < 32) pn = fmaf(-l, l, a[j + 1]);
        // column j of L to every lane (double-buffered: one warp barrier per column)
        float* cb = colbuf + (j & 1) * 32;
        cb[lane] = l;
        __syncwarp();
#pragma unroll
        for (int c4 = (j + 1) & ~3; c4 < 32; c4 += 4) {
          const float4 v = *reinterpret_cast<const float4*>(cb + c4);
          const float lc[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (c4 + e > j) a[c4 + e] = fmaf(-l, lc[e], a[c4 + e]);
        }
      }
#pragma unroll
      for (int c = 0; c < 32; c += 4)
        *reinterpret_cast<float4*>(row + c) =
            make_float4(c <= lane ? a[c] : 0.f, c + 1 <= lane ? a[c + 1] : 0.f,
                        c + 2 <= lane ? a[c + 2] : 0.f, c + 3 <= lane ? a[c + 3] : 0.f);
      rdiag[c0 + lane] = my_r;
      if (__any_sync(0xffffffffu, !(mypiv > 0.f))) bad = true;
#pragma unroll
      for (int c = 0; c < 32; ++c) LssT[c * LST + lane] = (c <= lane) ? a[c] : 0.f;
    }
    __syncthreads();
    // ---- T: rows below the sub-block, within the diagonal block (at most
    //      three warps), and the inverse of the diagonal sub-block (last warp)
    if (warp == FT / 32 - 1) invert_diag_block(s, Ls, rdiag, Mt, lane);
    if (t < b - c0 - 32) {
      float* row = Ls + (c0 + 32 + t) * LDM + c0;
      float a[32];
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 v = *reinterpret_cast<const float4*>(row + c);
        a[c] = v.x;
        a[c + 1] = v.y;
        a[c + 2] = v.z;
        a[c + 3] = v.w;
      }
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float x = a[c] * rdiag[c0 + c];
        a[c] = x;
        // column c of L_ss, read as rows of its transpose (broadcast loads)
#pragma unroll
        for (int m4 = (c + 1) & ~3; m4 < 32; m4 += 4) {
          const float4 v = *reinterpret_cast<const float4*>(LssT + c * LST + m4);
          const float lv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (m4 + e > c) a[m4 + e] = fmaf(-x, lv[e], a[m4 + e]);
        }
      }
#pragma unroll
      for (int c = 0; c < 32; c += 4)
        *reinterpret_cast<float4*>(row + c) = make_float4(a[c], a[c + 1], a[c + 2], a[c + 3]);
#pragma unroll
      for (int c = 0; c < 32; ++c) LT[c * LDM + c0 + 32 + t] = a[c];
    }
    __syncthreads();
    // ---- U: D_tu -= L_ts L_us^T for s < u <= t < nsub, 8 x 4 register tiles
    //      (one warp a 32 x 32 block) with both operands read along rows of
    //      the transposed sub-panel LT
    const int nt = nsub - s - 1;
    const int npairs = nt * (nt + 1) / 2;
    if (t < npairs * 32) {
      int pi = t >> 5;
      int tt = s + 1;
      while (pi > tt - s - 1) {  // pairs ordered (s+1,s+1), (s+2,s+1), (s+2,s+2), ...
        pi -= tt - s;
        ++tt;
      }
      const int uu = s + 1 + pi;
      const int i0 = 32 * tt + 8 * ((t >> 3) & 3), j0 = 32 * uu + 4 * (t & 7);
      float acc[8][4];
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
#pragma unroll 8
      for (int m = 0; m < 32; ++m) {
        const float4 x0 = *reinterpret_cast<const float4*>(LT + m * LDM + i0);
        const float4 x1 = *reinterpret_cast<const float4*>(LT + m * LDM + i0 + 4);
        const float4 y = *reinterpret_cast<const float4*>(LT + m * LDM + j0);
        const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w}, yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(xv[r], yv[c], acc[r][c]);
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        float4* o = reinterpret_cast<float4*>(Ls + (i0 + r) * LDM + j0);
        float4 v = *o;
        v.x -= acc[r][0];
        v.y -= acc[r][1];
        v.z -= acc[r][2];
        v.w -= acc[r][3];
        *o = v;
      }
    } else if (s >= 1 && t - npairs * 32 < s * 64) {
      // block row s of M, first half, with the threads the update leaves idle
      const int g = t - npairs * 32;
      inverse_rows_sum(s, g >> 6, g & 63, Ls, Mt, Tm);
    }
    __syncthreads();
  }
  // the last block row of M, second half
  if (nsub >= 2 && t < (nsub - 1) * 128) inverse_rows_finish(nsub - 1, t >> 7, t & 127, Tm, Mt);
  __syncthreads();
  return bad;
}

// Role products, RT = 1, 2 or 4 rows of the output per thread: lanes take
// the rows (lane + 32 i), warps take 8 output columns each (16 x 8 = 128).
//   X role: X_k[r][cb + c] = sum_q M[r][q] Acc[q][cb + c], r in this CTA's rows;
//   P role: P[rr][c] = sum_q A[rr][q] M[c][q], rr in this CTA's rows.
template <int RT>
__device__ __forceinline__ void role_products(const PanelArgs& p, bool xrole, int tile, int part,
                                              const float* __restrict__ Mt,
                                              const float* __restrict__ T, float* __restrict__ stg) {
  const int n = p.n, k = p.k, b = p.b;
  const int64_t ldz = n;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = 8 * warp;
  const int rows = 32 * RT;            // output rows of this CTA
  const int row0 = part * rows;        // first of them within the 128-row tile
  float acc[RT][8];
#pragma unroll
  for (int i = 0; i < RT; ++i)
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) acc[i][cc] = 0.f;
  if (xrole) {
    // Mt[q][r] = M[r][q] is zero for q > r, so q stops at the last row.
    const int cbase = tile * NB;
    const int qmax = min(b, row0 + rows);
    for (int q = 0; q < qmax; ++q) {
      const float4 t0 = *reinterpret_cast<const float4*>(T + q * LDM + c0);
      const float4 t1 = *reinterpret_cast<const float4*>(T + q * LDM + c0 + 4);
      const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
#pragma unroll
      for (int i = 0; i < RT; ++i) {
        const float m = Mt[q * LDM + row0 + lane + 32 * i];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) acc[i][cc] = fmaf(m, tv[cc], acc[i][cc]);
      }
    }
    const int w = min(NB, k - cbase);
    // B rows cbase + c, columns r: consecutive lanes, consecutive addresses.
    // The same values go to U row n-1-(k+r), columns n-1-cbase-c, through
    // shared memory so that consecutive lanes write consecutive columns.
#pragma unroll
    for (int i = 0; i < RT; ++i) {
      const int r = row0 + lane + 32 * i;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        stg[(lane + 32 * i) * LDM + c0 + cc] = acc[i][cc];
        if (r < b && c0 + cc < w)
          store_split(p.Bhi, p.Blo, static_cast<int64_t>(cbase + c0 + cc) * NB + r, acc[i][cc]);
      }
    }
    __syncthreads();
    const int nr = min(rows, b - row0);
    for (int idx = threadIdx.x; idx < nr * w; idx += PT) {
      const int rl = idx / w, c = idx - rl * w;
      p.U[static_cast<int64_t>(n - 1 - (k + row0 + rl)) * n + (n - 1 - cbase - c)] = stg[rl * LDM + c];
    }
  } else {
    // Mt[q][c] = M[c][q] is zero for q > c, so q stops after this warp's columns.
    const int rbase = k + b + tile * NB + row0;   // first panel row of this CTA
    const int h = min(rows, n - rbase);
    const int qmax = min(b, c0 + 8);
    for (int q = 0; q < qmax; q += 4) {
      float4 a4[RT];
#pragma unroll
      for (int i = 0; i < RT; ++i) a4[i] = *reinterpret_cast<const float4*>(T + (lane + 32 * i) * LDM + q);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float4 m0 = *reinterpret_cast<const float4*>(Mt + (q + e) * LDM + c0);
        const float4 m1 = *reinterpret_cast<const float4*>(Mt + (q + e) * LDM + c0 + 4);
        const float mv[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
        for (int i = 0; i < RT; ++i) {
          const float av = e == 0 ? a4[i].x : e == 1 ? a4[i].y : e == 2 ? a4[i].z : a4[i].w;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) acc[i][cc] = fmaf(av, mv[cc], acc[i][cc]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < RT; ++i) {
      const int rr = lane + 32 * i;
      if (rr >= h) continue;
      const int64_t off = static_cast<int64_t>(rbase + rr) * NB + c0;
      store_split4(p.Bhi, p.Blo, off, make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]));
      store_split4(p.Bhi, p.Blo, off + 4, make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]));
    }
    // this CTA's rows of the panel become the (zero) start of the Acc columns of block k
    __syncthreads();
    for (int idx = threadIdx.x; idx < h * (NB / 4); idx += PT) {
      const int rr = idx / (NB / 4), c4 = (idx % (NB / 4)) * 4;
      if (c4 < b)
        *reinterpret_cast<float4*>(p.Z + static_cast<int64_t>(rbase + rr) * ldz + k + c4) =
            make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// One step k of the factorization, in two kernels.
//   panel_factor_kernel (one CTA): factor the diagonal block and write
//     M^T = (L_kk^-1)^T to Mg.
//   panel_role_kernel: each CTA but the last takes `split` consecutive parts
//     (128/split rows) of one role tile: the Acc tiles left of the diagonal
//     block (X role), then the panel tiles below it (P role).  The last CTA
//     writes M itself: the diagonal block of U and B rows k..k+b.
// The factorization is the step's sequential chain, so it runs alone on one
// SM and writes only what the next kernel needs; the rest of the GPU stays
// free for the update GEMM of the previous step.
__global__ void __launch_bounds__(FT, 1) panel_factor_kernel(PanelArgs p) {
  extern __shared__ __align__(16) float sm[];
  float* Mt = sm;                    // [NB][LDM]  (L_kk^-1)^T
  float* Ls = Mt + NB * LDM;         // [NB][LDM]  diagonal block, then L_kk
  float* rdiag = Ls + NB * LDM;      // [NB]       1 / diag(L_kk)
  float* LT = rdiag + NB;            // [32][LDM] transposed sub-panel
  float* Tm = LT + 32 * LDM;         // [3][32][TMLD] partial sums of block rows of M
  float* colbuf = Tm + 3 * 32 * TMLD;  // [2][32]
  float* LssT = colbuf + 64;         // [32][LST] transposed diagonal sub-block
  const int t = threadIdx.x;
  for (int q = t; q < NB * (NB / 4); q += FT)
    *reinterpret_cast<float4*>(Mt + (q / (NB / 4)) * LDM + (q % (NB / 4)) * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
  // Launched with programmatic dependent launch.  The diagonal block comes
  // from the priority GEMM, which has completed once the kernel before this
  // one (the rest GEMM, which reads and writes neither the block nor what
  // this kernel writes) has let it in: then this kernel runs beside the rest
  // GEMM and waits for it only at its end (wait_first = 0).  Otherwise it
  // waits for the previous kernel first.  The role kernel is let in only at
  // the end, after that wait, so everything after this kernel is ordered
  // after the rest GEMM too; and its CTAs do not sit on SMs, waiting,
  // through the factorization.
  if (p.wait_first) griddep_wait();
  const bool notpd = factor_invert_blocked(p.Z, p.zlo, p.n, p.k, p.b, Mt, Ls, rdiag, Tm, LT, colbuf, LssT);
  if (t == 0 && notpd) atomicOr(p.status, kStatNotPD);
  __syncthreads();
  for (int idx = t; idx < NB * (NB / 4); idx += FT) {
    const int c = idx / (NB / 4), r4 = (idx % (NB / 4)) * 4;
    *reinterpret_cast<float4*>(p.Mg + c * NB + r4) = *reinterpret_cast<const float4*>(Mt + c * LDM + r4);
  }
  griddep_wait();
  griddep_launch_dependents();
}

__global__ void __launch_bounds__(PT, 1) panel_role_kernel(PanelArgs p) {
  extern __shared__ __align__(16) float sm[];
  float* Mt = sm;                    // [NB][LDM]  (L_kk^-1)^T
  float* T = Mt + NB * LDM;          // [NB][LDM]  role operand tile
  float* stg = T + NB * LDM;         // [NB][LDM]  X role: staged output rows
  const int n = p.n, k = p.k, b = p.b;
  const int64_t ldz = n;
  const int t = threadIdx.x;
  const bool diag_cta = blockIdx.x == gridDim.x - 1;
  const int tile = blockIdx.x / p.split;
  const int part = blockIdx.x % p.split;
  const bool xrole = tile < p.n_acc;
  const int ptile = tile - p.n_acc;  // P role: panel tile index
  const int prow = NB / p.split;     // rows of the P operand this CTA needs
  // Z, B and M come from the previous kernels.
  griddep_wait();
  griddep_launch_dependents();
  if (xrole && !diag_cta) {
    // The X role reads only its own rows of M: Mt[q][row0 .. row0 + rows).
    const int rows = NB / p.split, row0 = part * rows, n4 = rows / 4;
    for (int q = t; q < NB * n4; q += PT) {
      const int c = q / n4, r4 = row0 + (q % n4) * 4;
      cp_async16(Mt + c * LDM + r4, p.Mg + c * NB + r4, true);
    }
  } else {
    for (int q = t; q < NB * (NB / 4); q += PT) {
      const int c = q / (NB / 4), r4 = (q % (NB / 4)) * 4;
      cp_async16(Mt + c * LDM + r4, p.Mg + c * NB + r4, true);
    }
  }
  if (diag_cta) {
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    // X[k + r][k + c] = M[r][c] = Mt[c][r] for c <= r: U[n-1-k-r][n-1-k-c],
    // and B rows k..k+b (B[k + c][r] = Mt[c][r]).
    for (int idx = t; idx < NB * NB; idx += PT) {
      const int r = idx / NB, c = idx % NB;
      if (r < b && c <= r) p.U[static_cast<int64_t>(n - 1 - k - r) * n + (n - 1 - k - c)] = Mt[c * LDM + r];
    }
    for (int idx = t; idx < b * (NB / 4); idx += PT) {
      const int c = idx / (NB / 4), r4 = (idx % (NB / 4)) * 4;
      store_split4(p.Bhi, p.Blo, static_cast<int64_t>(k + c) * NB + r4,
                   *reinterpret_cast<const float4*>(Mt + c * LDM + r4));
    }
    return;
  }
  if (xrole) {  // T[q][cc] = Acc[k + q][cbase + cc], all 128 q
    const int cbase = tile * NB;
    for (int q = t; q < NB * (NB / 4); q += PT) {
      const int rr = q / (NB / 4), c4 = (q % (NB / 4)) * 4;
      const bool ok = rr < b && cbase + c4 < k;
      const float* src = p.Z + static_cast<int64_t>(k + rr) * ldz + cbase + c4;
      cp_async16(T + rr * LDM + c4, ok ? src : p.Z, ok);
    }
  } else {      // T[rr][q] = A[rbase + rr][k + q], this CTA's rows only
    const int rbase = k + b + ptile * NB + part * prow;
    for (int q = t; q < prow * (NB / 4); q += PT) {
      const int rr = q / (NB / 4), c4 = (q % (NB / 4)) * 4;
      const bool ok = rbase + rr < n && c4 < b;
      const float* src = p.Z + static_cast<int64_t>(rbase + rr) * ldz + k + c4;
      cp_async16(T + rr * LDM + c4, ok ? src : p.Z, ok);
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  if (p.split == 4)
    role_products<1>(p, xrole, xrole ? tile : ptile, part, Mt, T, stg);
  else if (p.split == 2)
    role_products<2>(p, xrole, xrole ? tile : ptile, part, Mt, T, stg);
  else
    role_products<4>(p, xrole, xrole ? tile : ptile, part, Mt, T, stg);
}

}  // namespace

// Workspace layout (byte offsets, each 256-aligned).
struct PrepLayout {
  size_t status, part, keys, zlo, Z, Mg, Bhi[2], Blo[2], total;
};

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

static PrepLayout prep_layout(int64_t d) {
  PrepLayout L;
  size_t off = 0;
  L.status = off;
  off += 256;
  L.part = off;  // fp64 sums of the diagonal, one per 256 entries
  off = align256(off + sizeof(double) * ((d + ST_THREADS - 1) / ST_THREADS));
  L.keys = off;
  off = align256(off + sizeof(unsigned long long) * d);
  L.zlo = off;
  off = align256(off + sizeof(float) * d);
  L.Z = off;
  off = align256(off + sizeof(float) * d * d);
  L.Mg = off;
  off = align256(off + sizeof(float) * NB * NB);
  for (int i = 0; i < 2; ++i) {  // panel operands of even and odd steps
    L.Bhi[i] = off;
    off = align256(off + sizeof(float) * d * NB);
    L.Blo[i] = off;
    off = align256(off + sizeof(float) * d * NB);
  }
  L.total = off;
  return L;
}

size_t prep_workspace_bytes(int64_t d) { return prep_layout(d).total; }

gptq_status_t launch_prepare(const float* S, const double* diag, int64_t d64, int64_t n_seen,
                             float damp, bool desc_act, float* U, int32_t* perm, void* ws,
                             cudaStream_t st) {
  const int d = static_cast<int>(d64);
  const PrepLayout L = prep_layout(d64);
  char* base = static_cast<char*>(ws);
  int* status = reinterpret_cast<int*>(base + L.status);
  double* part = reinterpret_cast<double*>(base + L.part);
  const int nparts = (d + ST_THREADS - 1) / ST_THREADS;
  auto* keys = reinterpret_cast<unsigned long long*>(base + L.keys);
  float* Z = reinterpret_cast<float*>(base + L.Z);
  float* zlo = reinterpret_cast<float*>(base + L.zlo);
  float* Mg = reinterpret_cast<float*>(base + L.Mg);
  const double hscale = 2.0 / static_cast<double>(n_seen);

  GPTQ_CUDA_TRY(cudaMemsetAsync(status, 0, sizeof(int), st));
  prep_stats_kernel<<<nparts, ST_THREADS, 0, st>>>(S, diag, d, keys, part, desc_act ? nullptr : perm,
                                                   status);
  GPTQ_LAUNCH_CHECK();
  if (desc_act) {
    prep_rank_kernel<<<(d + 255) / 256, 256, 0, st>>>(keys, d, perm);
    GPTQ_LAUNCH_CHECK();
  }
  {
    dim3 grid((d + 31) / 32, (d + 31) / 32), block(32, 8);
    prep_gather_kernel<<<grid, block, 0, st>>>(S, perm, d, static_cast<float>(hscale), Z, U, status);
    GPTQ_LAUNCH_CHECK();
    prep_diag_kernel<<<(d + 255) / 256, 256, 0, st>>>(S, diag, perm, d, hscale, damp, part, nparts, Z, zlo,
                                                      status);
    GPTQ_LAUNCH_CHECK();
  }
  const size_t smem_factor = sizeof(float) * (2 * NB * LDM + NB + 32 * LDM + 3 * 32 * TMLD + 64 + 32 * LST);
  const size_t smem_role = sizeof(float) * (3 * NB * LDM);
  GPTQ_CUDA_TRY(cudaFuncSetAttribute(panel_factor_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem_factor)));
  GPTQ_CUDA_TRY(cudaFuncSetAttribute(panel_role_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem_role)));
  const int sms = sm_count();

  // Step k: factor the diagonal block (one CTA), the role products, then the
  // update of the trailing rows by B_k in two launches on this stream: the
  // "priority" tiles (the next step's row block and column block, all that
  // step k + 1's factor and role kernels read), then the "rest" on all SMs
  // but one.  Step k + 1's factor kernel starts beside the rest GEMM on the
  // SM it leaves free (see panel_factor_kernel), and every later kernel is
  // still ordered after the rest GEMM.  The panel operand B alternates
  // between two buffers by step parity.
  gptq_status_t result = GPTQ_OK;
  bool after_rest = false;  // the last kernel launched is a rest GEMM
  for (int k = 0; k < d && result == GPTQ_OK; k += NB) {
    const int b = std::min(NB, d - k);
    const int par = (k / NB) & 1;
    float* Bhi = reinterpret_cast<float*>(base + L.Bhi[par]);
    float* Blo = reinterpret_cast<float*>(base + L.Blo[par]);
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
    pa.zlo = zlo;
    pa.Mg = Mg;
    pa.wait_first = after_rest ? 0 : 1;
    const int n_pan = (d - k - b + NB - 1) / NB;
    const int tiles = pa.n_acc + n_pan;
    pa.split = (4 * tiles < sms) ? 4 : (2 * tiles < sms) ? 2 : 1;
    count_launch();
    if (cudaSuccess != launch_pdl(panel_factor_kernel, dim3(1), dim3(FT), smem_factor, st, pa) ||
        cudaSuccess != cudaGetLastError()) {
      result = GPTQ_ERR_CUDA;
      break;
    }
    count_launch();
    if (cudaSuccess != launch_pdl(panel_role_kernel, dim3(tiles * pa.split + 1), dim3(PT), smem_role, st,
                                  pa) ||
        cudaSuccess != cudaGetLastError()) {
      result = GPTQ_ERR_CUDA;
      break;
    }
    after_rest = false;
    if (k + b >= d) break;
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
    g.diag_lo = zlo;
    g.pri_nt = (k + b) / NB;
    const float* Ahi = Bhi + static_cast<int64_t>(k + b) * NB;
    const float* Alo = Blo + static_cast<int64_t>(k + b) * NB;
    g.subset = 1;
    result = launch_tgemm_3xtf32(Ahi, Alo, NB, Bhi, Blo, NB, g, status, st);
    if (result != GPTQ_OK) break;
    g.subset = 2;
    if (tgemm_tile_count(g) == 0) continue;
    g.max_ctas = sms - 1;  // the free SM takes the next factor kernel
    result = launch_tgemm_3xtf32(Ahi, Alo, NB, Bhi, Blo, NB, g, status, st);
    after_rest = true;
  }
  return result;
}

}  // namespace gptq
