// 3xTF32 GEMM on tcgen05 (see tgemm.cuh for the contract).
//
// Structure (one CTA per SM, persistent over output tiles of 128 x BN,
// BN = 128, or 64 for launches that would fill fewer than half the SMs: the
// tiles then halve and the CTAs double, and each tile's latency shrinks):
//   warp 0      TMA producer: per 32-wide K slab, the fp32 tiles A_hi, A_lo
//               (128 x 32) and B_hi, B_lo (BN x 32) into a 3-stage (BN = 128)
//               or 4-stage (BN = 64) ring, 128-byte swizzle
//   warp 1      MMA issuer: per K slab, 4 steps of K=8, each three
//               tcgen05.mma kind::tf32 (lo*hi, hi*lo, hi*hi) into TMEM
//   warps 2-9   epilogue: TMEM -> registers -> C = alpha*acc + beta*C
// Two BN-column TMEM accumulators let the epilogue of one tile overlap the
// MMAs of the next.
#include <algorithm>
#include <atomic>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "tgemm.cuh"

namespace gptq {
namespace {

constexpr int BM = 128;
constexpr int BK = 32;  // fp32: 128 bytes per row = one swizzle span
constexpr int UK = 8;   // K of one kind::tf32 MMA
constexpr int A_TILE = BM * BK * 4;  // 16 KB
constexpr int NUM_THREADS = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue

template <int BN>
struct TCfg {
  static constexpr int STAGES = BN == 64 ? 4 : 3;
  static constexpr int B_TILE = BN * BK * 4;
  static constexpr int STAGE_BYTES = 2 * A_TILE + 2 * B_TILE;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static constexpr int PR = 128 / BN;  // tiles of one 128-column priority block
};

struct TGemmSched {
  int m_tiles, n_tiles, k_blocks, tiles;
};

// Tiles of tile row mt below or on the diagonal (all of them without `lower`).
template <int BN>
__host__ __device__ __forceinline__ int row_tiles(const TGemmArgs& a, int n_tiles, int mt) {
  if (!a.lower) return n_tiles;
  const long long lim = static_cast<long long>(a.row_off) + static_cast<long long>(mt) * BM + BM - 1 -
                        a.col_off;
  if (lim < 0) return 0;
  return static_cast<int>(lim / BN + 1 < n_tiles ? lim / BN + 1 : n_tiles);
}

// Tiles of row mt inside the priority block of columns [128 pri_nt, + 128).
template <int BN>
__host__ __device__ __forceinline__ int pri_tiles(const TGemmArgs& a, int c) {
  const int lo = a.pri_nt * TCfg<BN>::PR;
  const int n = c - lo;
  return n <= 0 ? 0 : (n < TCfg<BN>::PR ? n : TCfg<BN>::PR);
}

// Tiles of row mt in the launch's subset.
template <int BN>
__host__ __device__ __forceinline__ int subset_row_tiles(const TGemmArgs& a, int n_tiles, int mt) {
  const int c = row_tiles<BN>(a, n_tiles, mt);
  if (a.subset == 0) return c;
  const int np = pri_tiles<BN>(a, c);
  if (a.subset == 1) return mt == 0 ? c : np;
  return mt == 0 ? 0 : c - np;
}

// The t-th tile of the subset, rows in order, columns in order within a row.
template <int BN>
__host__ __device__ __forceinline__ void tile_coords(const TGemmArgs& a, const TGemmSched& s, int t, int& mt,
                                            int& nt) {
  for (mt = 0; mt < s.m_tiles; ++mt) {
    const int c = subset_row_tiles<BN>(a, s.n_tiles, mt);
    if (t < c) break;
    t -= c;
  }
  const int lo = a.pri_nt * TCfg<BN>::PR;
  if (a.subset == 1 && mt > 0)
    nt = lo + t;
  else if (a.subset == 2 && mt > 0 && t >= lo)
    nt = t + pri_tiles<BN>(a, row_tiles<BN>(a, s.n_tiles, mt));
  else
    nt = t;
}

// PAIR: clusters of two CTAs take the vertically adjacent tiles (2p, nt) and
// (2p + 1, nt) of a full (non-triangular, all-tiles) update; they share the
// tile's B rows, so each CTA loads its own A and one half of B, multicast to
// both (TMA multicast within this GPU's memory): 48 KB of L2 reads per
// 32-wide K slab and CTA instead of 64 KB.  A slot is free again once both
// CTAs' MMAs have read it: each MMA thread releases it in both CTAs with one
// multicast commit.
template <int BN, bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tgemm_kernel(const __grid_constant__ CUtensorMap tm_ahi, const __grid_constant__ CUtensorMap tm_alo,
                 const __grid_constant__ CUtensorMap tm_bhi, const __grid_constant__ CUtensorMap tm_blo,
                 TGemmArgs a, TGemmSched s, int* fault) {
  constexpr int STAGES = TCfg<BN>::STAGES;
  constexpr int STAGE_BYTES = TCfg<BN>::STAGE_BYTES;
  constexpr int B_TILE = TCfg<BN>::B_TILE;
  constexpr uint32_t TMEM_COLS = TCfg<BN>::TMEM_COLS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int i) { return bar0 + 8u * i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (STAGES + i); };
  auto accf_bar = [&](int i) { return bar0 + 8u * (2 * STAGES + i); };
  auto acce_bar = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 + i); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const int cid = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int nclusters = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  // the tile of job t: in PAIR mode, pair row block t / n_tiles, column t % n_tiles
  auto job_tile = [&](int t, int& mt, int& nt) {
    if constexpr (PAIR) {
      mt = 2 * (t / s.n_tiles) + rank;
      nt = t % s.n_tiles;
    } else {
      tile_coords<BN>(a, s, t, mt, nt);
    }
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), PAIR ? 2 : 1);   // PAIR: released by both CTAs' MMAs
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(accf_bar(i), 1);
      mbar_init(acce_bar(i), 256);
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_ahi);
    tma_prefetch_desc(&tm_alo);
    tma_prefetch_desc(&tm_bhi);
    tma_prefetch_desc(&tm_blo);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync();   // both CTAs' barriers exist before either multicasts into the other
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Everything above is independent of the previous kernel (launched with
  // programmatic dependent launch); A, B and C are not.
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = cid; ok && t < s.tiles; t += nclusters) {
        int mt, nt;
        job_tile(t, mt, nt);
        for (int kb = 0; kb < s.k_blocks; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, fault)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          tma_load_2d(sa, &tm_ahi, fb, kb * BK, mt * BM);
          tma_load_2d(sa + A_TILE, &tm_alo, fb, kb * BK, mt * BM);
          if constexpr (PAIR) {  // own half of B, to both CTAs; the other half comes from the peer
            tma_load_2d_multicast(sa + 2 * A_TILE + rank * (B_TILE / 2), &tm_bhi, fb, kb * BK,
                                  nt * BN + rank * (BN / 2), 0x3);
            tma_load_2d_multicast(sa + 2 * A_TILE + B_TILE + rank * (B_TILE / 2), &tm_blo, fb, kb * BK,
                                  nt * BN + rank * (BN / 2), 0x3);
          } else {
            tma_load_2d(sa + 2 * A_TILE, &tm_bhi, fb, kb * BK, nt * BN);
            tma_load_2d(sa + 2 * A_TILE + B_TILE, &tm_blo, fb, kb * BK, nt * BN);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if constexpr (PAIR) {
        // Before this CTA may exit, every release the peer sends to its
        // slots must have landed: wait for one more turn of the ring.
        for (int i = 0; i < STAGES; ++i) {
          mbar_wait_bounded(empty_bar(stage), phase ^ 1u, fault);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(BM, BN, /*tf32*/ 2, /*tf32*/ 2);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int t = cid; ok && t < s.tiles; t += nclusters) {
        if (!mbar_wait_bounded(acce_bar(acc), acc_phase ^ 1u, fault)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < s.k_blocks; ++kb) {
          if (!mbar_wait_bounded(full_bar(stage), phase, fault)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint64_t d_ahi = smem_desc_sw128_kmajor(sa);
          const uint64_t d_alo = smem_desc_sw128_kmajor(sa + A_TILE);
          const uint64_t d_bhi = smem_desc_sw128_kmajor(sa + 2 * A_TILE);
          const uint64_t d_blo = smem_desc_sw128_kmajor(sa + 2 * A_TILE + B_TILE);
#pragma unroll
          for (int k = 0; k < BK / UK; ++k) {
            const uint64_t off = static_cast<uint64_t>((k * UK * 4) >> 4);  // 32 bytes per step
            const uint32_t first = (kb == 0 && k == 0) ? 0u : 1u;
            tc_mma_tf32(d_tmem, d_alo + off, d_bhi + off, idesc, first);
            tc_mma_tf32(d_tmem, d_ahi + off, d_blo + off, idesc, 1u);
            tc_mma_tf32(d_tmem, d_ahi + off, d_bhi + off, idesc, 1u);
          }
          if constexpr (PAIR)
            tc_commit_multicast(empty_bar(stage), 0x3);  // frees the slot in both CTAs
          else
            tc_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(accf_bar(acc));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      tc_commit(drain_bar);
      mbar_wait_bounded(drain_bar, 0, fault);
    }
  } else {
    // Epilogue, 8 warps: warp w reads TMEM lanes 32q..32q+31 (q = w mod 4,
    // the quarter it may access) and columns 64h..64h+63 of the tile
    // (h = 0 for warps 2-5, 1 for warps 6-9); each lane owns one row.  The
    // row's C values are loaded before the accumulator is waited for, so
    // the read latency overlaps the tile's MMAs.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = cid; t < s.tiles; t += nclusters) {
      int mt, nt;
      job_tile(t, mt, nt);
      const int m = mt * BM + q * 32 + lane;
      const bool row_ok = m < a.M;
      const long long diag = static_cast<long long>(a.row_off) + m - a.col_off;  // n <= diag
      float* crow = a.C + static_cast<int64_t>(m) * a.ldc;
      constexpr int NCH = BN / 64;    // 32-column chunks of this warp's half of the tile
      // Every C value the chunk will update (and the diagonal one, for the
      // two-sum) is loaded here, before the wait: the loads of a chunk that
      // the diagonal or the matrix edge cuts are scalar but just as early,
      // instead of one dependent load-store pair per element after it.
      const bool need_c = a.beta != 0.f || a.diag_lo != nullptr;
      float cpre[NCH][32];
      bool fast[NCH];
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) {
        const int n0 = nt * BN + h * (BN / 2) + cc * 32;
        fast[cc] = row_ok && (n0 + 32 <= a.N) && (!a.lower || n0 + 31 <= diag) && (a.ldc % 4 == 0);
        if (fast[cc]) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 x = need_c ? *reinterpret_cast<const float4*>(crow + n0 + 4 * i)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            cpre[cc][4 * i] = x.x;
            cpre[cc][4 * i + 1] = x.y;
            cpre[cc][4 * i + 2] = x.z;
            cpre[cc][4 * i + 3] = x.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int n = n0 + i;
            const bool ok = need_c && row_ok && n < a.N && (!a.lower || n <= diag);
            cpre[cc][i] = ok ? crow[n] : 0.f;
          }
        }
      }
      if (!mbar_wait_bounded(accf_bar(acc), acc_phase, fault)) break;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) {
        const int n0 = nt * BN + h * (BN / 2) + cc * 32;
        if (n0 < a.N) {  // warp-uniform
        float v[32];
        tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                               static_cast<uint32_t>(acc * BN + h * (BN / 2) + cc * 32),
                           v);
        if (row_ok && a.diag_lo && diag >= n0 && diag < n0 + 32 && diag < a.N) {
          // the diagonal element of this row lies in the chunk: two-sum
          const int i = static_cast<int>(diag - n0);
          float vi = 0.f, cv = 0.f;  // v[i], C[diag] without a dynamic index (keeps them in registers)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            vi = (e == i) ? v[e] : vi;
            cv = (e == i) ? cpre[cc][e] : cv;
          }
          const float tt = -vi;
          const float sum = cv + tt;
          const float bb = sum - cv;
          const float err = (cv - (sum - bb)) + (tt - bb);
          a.diag_lo[a.col_off + diag] += err;
        }
        if (row_ok && fast[cc]) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float4 o = make_float4(a.alpha * v[4 * i], a.alpha * v[4 * i + 1], a.alpha * v[4 * i + 2],
                                   a.alpha * v[4 * i + 3]);
            if (a.beta != 0.f) {
              o.x = fmaf(a.beta, cpre[cc][4 * i], o.x);
              o.y = fmaf(a.beta, cpre[cc][4 * i + 1], o.y);
              o.z = fmaf(a.beta, cpre[cc][4 * i + 2], o.z);
              o.w = fmaf(a.beta, cpre[cc][4 * i + 3], o.w);
            }
            *reinterpret_cast<float4*>(crow + n0 + 4 * i) = o;
          }
        } else if (row_ok) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int n = n0 + i;
            if (n >= a.N || (a.lower && n > diag)) continue;
            float o = a.alpha * v[i];
            if (a.beta != 0.f) o = fmaf(a.beta, cpre[cc][i], o);
            crow[n] = o;
          }
        }
        }
      }
      tc_fence_before();
      mbar_arrive(acce_bar(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync();   // neither CTA leaves while the other may still use its shared memory
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool make_f32_map(CUtensorMap* m, const float* base, int64_t rows, int64_t k, int64_t ld, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
  cuuint32_t box[2] = {BK, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN>
TGemmSched make_sched(const TGemmArgs& a) {
  TGemmSched s;
  s.m_tiles = (a.M + BM - 1) / BM;
  s.n_tiles = (a.N + BN - 1) / BN;
  s.k_blocks = (a.K + BK - 1) / BK;
  s.tiles = 0;
  for (int mt = 0; mt < s.m_tiles; ++mt) s.tiles += subset_row_tiles<BN>(a, s.n_tiles, mt);
  return s;
}

template <int BN, bool PAIR>
gptq_status_t launch_bn(const float* A_hi, const float* A_lo, int64_t lda, const float* B_hi,
                        const float* B_lo, int64_t ldb, const TGemmArgs& args, const TGemmSched& s,
                        int* fault, cudaStream_t st) {
  CUtensorMap m_ahi, m_alo, m_bhi, m_blo;
  const int b_rows = PAIR ? BN / 2 : BN;   // PAIR: each CTA loads half of B
  if (!make_f32_map(&m_ahi, A_hi, args.M, args.K, lda, BM) ||
      !make_f32_map(&m_alo, A_lo, args.M, args.K, lda, BM) ||
      !make_f32_map(&m_bhi, B_hi, args.N, args.K, ldb, b_rows) ||
      !make_f32_map(&m_blo, B_lo, args.N, args.K, ldb, b_rows))
    return GPTQ_ERR_CUDA;
  // The shared-memory attribute is set once per device (two threads that
  // race here both set the same value).
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  GPTQ_CUDA_TRY(cudaGetDevice(&dev));
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (!bit || !(attr_set.load(std::memory_order_relaxed) & bit)) {
    GPTQ_CUDA_TRY(cudaFuncSetAttribute(tgemm_kernel<BN, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TCfg<BN>::SMEM_BYTES));
    attr_set.fetch_or(bit, std::memory_order_relaxed);
  }
  if constexpr (PAIR) {
    // one cluster of two CTAs per tile pair in flight, launched like launch_pdl
    int clusters = std::min(sm_count() / 2, s.tiles);
    if (args.max_ctas > 0) clusters = std::min(clusters, std::max(1, args.max_ctas / 2));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = TCfg<BN>::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    GPTQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, tgemm_kernel<BN, PAIR>, m_ahi, m_alo, m_bhi, m_blo, args, s,
                                     fault));
  } else {
    int grid = std::min(sm_count(), s.tiles);
    if (args.max_ctas > 0) grid = std::min(grid, args.max_ctas);
    GPTQ_CUDA_TRY(launch_pdl(tgemm_kernel<BN, PAIR>, dim3(grid), dim3(NUM_THREADS), TCfg<BN>::SMEM_BYTES,
                             st, m_ahi, m_alo, m_bhi, m_blo, args, s, fault));
  }
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

}  // namespace

int tgemm_tile_count(const TGemmArgs& args) { return make_sched<128>(args).tiles; }

// A launch that would fill fewer than half the SMs with 128 x 128 tiles runs
// 128 x 64 tiles: twice the CTAs, each tile's loads, MMAs and epilogue about
// half.
static bool narrow_tiles(int tiles128, int sms) { return 2 * tiles128 <= sms; }

// The tiles of one launch for a GPU with `sms` SMs, in the order its CTAs
// take them (tile row, tile column); returns the count and the tile width.
template <int BN>
static int list_tiles(const TGemmArgs& a, int32_t* coords, int cap) {
  const TGemmSched s = make_sched<BN>(a);
  for (int t = 0; t < s.tiles && t < cap; ++t) {
    int mt, nt;
    tile_coords<BN>(a, s, t, mt, nt);
    coords[2 * t] = mt;
    coords[2 * t + 1] = nt;
  }
  return s.tiles;
}

int tgemm_plan(const TGemmArgs& a, int sms, int* bn, int32_t* coords, int cap) {
  const TGemmSched s = make_sched<128>(a);
  if (s.tiles > 0 && narrow_tiles(s.tiles, sms)) {
    *bn = 64;
    return list_tiles<64>(a, coords, cap);
  }
  *bn = 128;
  return list_tiles<128>(a, coords, cap);
}

gptq_status_t launch_tgemm_3xtf32(const float* A_hi, const float* A_lo, int64_t lda, const float* B_hi,
                                  const float* B_lo, int64_t ldb, const TGemmArgs& args, int* fault,
                                  cudaStream_t st) {
  if (!fault) return GPTQ_ERR_CUDA;
  if (args.M <= 0 || args.N <= 0 || args.K <= 0) return GPTQ_OK;
  const TGemmSched s = make_sched<128>(args);
  if (s.tiles == 0) return GPTQ_OK;
  if (narrow_tiles(s.tiles, sm_count())) {
    const TGemmSched s64 = make_sched<64>(args);
    return launch_bn<64, false>(A_hi, A_lo, lda, B_hi, B_lo, ldb, args, s64, fault, st);
  }
  if (args.subset == 0 && !args.lower) {
    // A full rectangular update: tile pairs sharing their B rows (the jobs
    // are the pairs; an odd last tile row pairs with rows beyond M, which
    // the TMA fills with zeros and the epilogue does not write).
    TGemmSched sp = s;
    sp.tiles = ((s.m_tiles + 1) / 2) * s.n_tiles;
    return launch_bn<128, true>(A_hi, A_lo, lda, B_hi, B_lo, ldb, args, sp, fault, st);
  }
  return launch_bn<128, false>(A_hi, A_lo, lda, B_hi, B_lo, ldb, args, s, fault, st);
}

}  // namespace gptq

// Test hook (not part of the public header): C = alpha A B^T + beta C with
// A, B given as TF32 hi/lo pairs, on `stream`.
extern "C" GPTQ_API int gptq_internal_tgemm(const float* A_hi, const float* A_lo, int64_t lda,
                                            const float* B_hi, const float* B_lo, int64_t ldb, int M,
                                            int N, int K, float alpha, float beta, float* C,
                                            int64_t ldc, int lower, int row_off, int col_off,
                                            gptq_stream_t stream) {
  gptq::TGemmArgs g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.alpha = alpha;
  g.beta = beta;
  g.C = C;
  g.ldc = ldc;
  g.lower = lower;
  g.row_off = row_off;
  g.col_off = col_off;
  return gptq::launch_tgemm_3xtf32(A_hi, A_lo, lda, B_hi, B_lo, ldb, g, gptq::fault_word_ptr(),
                                   reinterpret_cast<cudaStream_t>(stream));
}

// Test hook (not part of the public header): the same update restricted to
// one tile subset (0 all, 1 the first tile row and tile column pri_nt, 2 the
// others), on at most max_ctas CTAs (0: one per SM).
extern "C" GPTQ_API int gptq_internal_tgemm_subset(const float* A_hi, const float* A_lo, int64_t lda,
                                                   const float* B_hi, const float* B_lo, int64_t ldb,
                                                   int M, int N, int K, float alpha, float beta,
                                                   float* C, int64_t ldc, int lower, int row_off,
                                                   int col_off, int subset, int pri_nt, int max_ctas,
                                                   int* tiles, gptq_stream_t stream) {
  if (subset < 0 || subset > 2 || pri_nt < 0 || max_ctas < 0) return GPTQ_ERR_INVALID_ARG;
  gptq::TGemmArgs g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.alpha = alpha;
  g.beta = beta;
  g.C = C;
  g.ldc = ldc;
  g.lower = lower;
  g.row_off = row_off;
  g.col_off = col_off;
  g.subset = subset;
  g.pri_nt = pri_nt;
  g.max_ctas = max_ctas;
  if (tiles) *tiles = gptq::tgemm_tile_count(g);
  return gptq::launch_tgemm_3xtf32(A_hi, A_lo, lda, B_hi, B_lo, ldb, g, gptq::fault_word_ptr(),
                                   reinterpret_cast<cudaStream_t>(stream));
}

// Test hook (not part of the public header), host only: the tiles one update
// launch of the given subset would take on a GPU with `sms` SMs, as (tile
// row, tile column) pairs in the order the CTAs take them (at most cap
// pairs written), and the tile width it would use (*bn: 64 or 128; tiles are
// 128 rows high).  A full rectangular update runs the same 128 x 128 tiles
// in vertically adjacent pairs.  Returns the tile count, or -1 for bad
// arguments.  Nothing is launched.
extern "C" GPTQ_API int gptq_internal_tgemm_tiles(int M, int N, int lower, int row_off, int col_off,
                                                  int subset, int pri_nt, int sms, int* bn,
                                                  int32_t* coords, int cap) {
  if (M <= 0 || N <= 0 || subset < 0 || subset > 2 || pri_nt < 0 || sms <= 0 || !bn || cap < 0 ||
      (cap > 0 && !coords))
    return -1;
  gptq::TGemmArgs g;
  g.M = M;
  g.N = N;
  g.K = 128;
  g.lower = lower;
  g.row_off = row_off;
  g.col_off = col_off;
  g.subset = subset;
  g.pri_nt = pri_nt;
  return gptq::tgemm_plan(g, sms, bn, coords, cap);
}
