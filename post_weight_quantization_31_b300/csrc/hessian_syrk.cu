// Step a1: S += X X^T on the 5th-generation tensor cores.
//
// [G] GPTQ practical guide (m.lqnn.cn/news/117696), §2.1: the Hessian is
// computed from the calibration activations of the layer; the guide (and the
// "tens of minutes" figures of the ms-swift review) place most of the time in
// this per-layer Hessian work.  H = 2/n S is formed later, in a2.
//
// Design (sm_103a):
//   * S is symmetric, so only output tiles that touch the upper triangle
//     (row <= col) are computed: 128 x 256 tiles (UMMA M=128, N=256,
//     cta_group::1), A = X[rows of the tile, k-slab], B = X[cols of the
//     tile, k-slab]; both K-major, fp16 x fp16 -> fp32 in TMEM.
//   * Operands are staged by TMA (128-byte swizzle, 64 tokens per stage)
//     through a 4-stage mbarrier ring; one thread issues tcgen05.mma, one
//     thread issues TMA, eight warps drain the accumulators.
//   * X may be channel-major ([d, n_tok], tokens contiguous: K-major
//     operands, one box of 128 or 256 channels x 64 tokens per operand) or
//     token-major ([n_tok, d], channels contiguous: MN-major operands, boxes
//     of 64 channels x 64 tokens, two for A and four for B, which the MMA
//     reads through MN-major descriptors).  Same tiles, same schedule.
//   * Two 256-column TMEM accumulators (all 512 columns).  The tensor cores
//     add into an accumulator with a rounding that is biased over long
//     chains (measured: S_ii 0.15% low after 262144 tokens), so one
//     accumulator takes at most CH slabs (1024 tokens); eight drain warps then
//     add it into fp32 registers with round-to-nearest while the MMAs fill
//     the other accumulator.  A job's sum leaves the registers once, at its
//     end.
//   * CTAs run in clusters of two that take the two tiles (ti, tj) and
//     (ti + 1, tj) of one column block: they share the tile's 256 B rows,
//     so each CTA loads its own A and one half of B, multicast to both
//     (TMA multicast within this GPU's memory).  A 64-token stage then costs
//     each CTA 32 KB of L2 reads instead of 48 KB; the MMAs are unchanged
//     (one CTA, M = 128).  A stage slot is free again once both CTAs' MMAs
//     have read it: each MMA thread releases it in both CTAs with one
//     multicast commit.
//   * Jobs: whole tile pairs with the full token range first, in waves of
//     one pair per cluster (every cluster of a wave sweeps the tokens at the
//     same pace, so each X slab is read from HBM about once per wave and
//     re-served from L2); the pairs left over after the last full wave are
//     split along the tokens into `ks` pieces to balance the final wave.
//   * Results are added to S with fp32 atomics: element (r, c), r <= c, goes
//     to S[r][c] and, for r < c, also to S[c][r].
#include <algorithm>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace gptq {
namespace {

constexpr int BM = 128;             // tile rows (UMMA M)
constexpr int BN = 256;             // tile cols (UMMA N)
constexpr int BK = 64;              // tokens per stage: 128 bytes of fp16
constexpr int UK = 16;              // K of one tcgen05.mma kind::f16
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 320;    // warp 0 TMA, warp 1 MMA, warps 2-9 drain
constexpr int CH = 16;              // slabs (BK tokens each) per accumulator fill
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
constexpr uint32_t TMEM_COLS = 512;

struct SyrkSchedule {
  int d;         // d_col
  int kb_total;  // token slabs of BK
  int n_i;       // row blocks of BM
  int tiles;     // tiles touching the upper triangle
  int pairs;     // tile pairs (row blocks 2m, 2m + 1 of one column block)
  int full;      // jobs covering a whole pair (multiple of the clusters)
  int rem;       // pairs split into pieces
  int ks;        // pieces per split pair
  int jobs;
};

// Column block tj of 256 holds the row blocks ti < min(n_i, 2 tj + 2):
// ceil(that / 2) pairs.  Pair p -> (first row block ti0 = 2m, tj).  With an
// odd count the pair's second tile lies past d (row block n_i) and adds
// nothing.
__device__ __forceinline__ void pair_of(int p, int n_i, int& ti0, int& tj) {
  int j = 0;
  for (;;) {
    const int c = (min(n_i, 2 * j + 2) + 1) / 2;
    if (p < c) break;
    p -= c;
    ++j;
  }
  ti0 = 2 * p;
  tj = j;
}

__device__ __forceinline__ void job_of(const SyrkSchedule& s, int job, int& ti0, int& tj, int& k0,
                                       int& k1) {
  int pair;
  if (job < s.full) {
    pair = job;
    k0 = 0;
    k1 = s.kb_total;
  } else {
    const int jj = job - s.full;
    const int piece = jj / s.rem;
    pair = s.full + jj % s.rem;
    k0 = static_cast<int>(static_cast<long long>(piece) * s.kb_total / s.ks);
    k1 = static_cast<int>(static_cast<long long>(piece + 1) * s.kb_total / s.ks);
  }
  pair_of(pair, s.n_i, ti0, tj);
}

// Token-major boxes: 64 channels (128 bytes) x BK tokens = 8 KB each.
constexpr int TM_BOX = 64;
constexpr int TM_BOX_BYTES = TM_BOX * BK * 2;

template <bool TOKMAJOR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    hessian_syrk_kernel(const __grid_constant__ CUtensorMap tm_a,
                        const __grid_constant__ CUtensorMap tm_b, SyrkSchedule s, float* __restrict__ S,
                        int* fault) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  // bars[0..S): full, [S..2S): empty, [2S..2S+2): acc full, [2S+2..2S+4): acc empty,
  // [2S+4]: drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int i) { return bar0 + 8u * i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (STAGES + i); };
  auto accf_bar = [&](int i) { return bar0 + 8u * (2 * STAGES + i); };
  auto acce_bar = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 + i); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int rank = static_cast<int>(cluster_ctarank());   // 0 or 1 within the pair
  const int cid = blockIdx.x >> 1, nclusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), 2);   // released by both CTAs' MMAs
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(accf_bar(i), 1);
      mbar_init(acce_bar(i), 256);
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();   // both CTAs' barriers exist before either multicasts into the other
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int job = cid; ok && job < s.jobs; job += nclusters) {
        int ti0, tj, k0, k1;
        job_of(s, job, ti0, tj, k0, k1);
        const int ti = ti0 + rank;
        for (int kb = k0; kb < k1; ++kb) {
          // the slot is free once both CTAs' MMAs have read it
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, fault)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          // own A, own half of B to both CTAs; the other half comes from the peer
          mbar_arrive_expect_tx(full_bar(stage), STAGE_BYTES);
          if constexpr (TOKMAJOR) {
#pragma unroll
            for (int c = 0; c < BM / TM_BOX; ++c)
              tma_load_2d(sa + c * TM_BOX_BYTES, &tm_a, full_bar(stage), ti * BM + c * TM_BOX, kb * BK);
#pragma unroll
            for (int c = rank * (BN / TM_BOX / 2); c < (rank + 1) * (BN / TM_BOX / 2); ++c)
              tma_load_2d_multicast(sa + A_BYTES + c * TM_BOX_BYTES, &tm_b, full_bar(stage),
                                    tj * BN + c * TM_BOX, kb * BK, 0x3);
          } else {
            tma_load_2d(sa, &tm_a, full_bar(stage), kb * BK, ti * BM);
            tma_load_2d_multicast(sa + A_BYTES + rank * (B_BYTES / 2), &tm_b, full_bar(stage), kb * BK,
                                  tj * BN + rank * (BN / 2), 0x3);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Before this CTA may exit, every release the peer sends to its slots
      // must have landed: wait for one more turn of the ring.
      for (int i = 0; i < STAGES; ++i) {
        mbar_wait_bounded(empty_bar(stage), phase ^ 1u, fault);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(BM, BN, /*a f16*/ 0, /*b f16*/ 0, TOKMAJOR ? 1 : 0,
                                            TOKMAJOR ? 1 : 0);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int job = cid; ok && job < s.jobs; job += nclusters) {
        int ti0, tj, k0, k1;
        job_of(s, job, ti0, tj, k0, k1);
        for (int c0 = k0; ok && c0 < k1; c0 += CH) {
          const int c1 = min(k1, c0 + CH);
          if (!mbar_wait_bounded(acce_bar(acc), acc_phase ^ 1u, fault)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
          for (int kb = c0; kb < c1; ++kb) {
            if (!mbar_wait_bounded(full_bar(stage), phase, fault)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
            uint64_t da, db;
            if constexpr (TOKMAJOR) {
              // 64-channel chunks 8 KB apart, 8-token groups 1 KB apart.
              da = smem_desc_sw128_mnmajor(sa, TM_BOX_BYTES, 1024);
              db = smem_desc_sw128_mnmajor(sa + A_BYTES, TM_BOX_BYTES, 1024);
            } else {
              da = smem_desc_sw128_kmajor(sa);
              db = smem_desc_sw128_kmajor(sa + A_BYTES);
            }
#pragma unroll
            for (int k = 0; k < BK / UK; ++k) {
              // K-major: advance 32 bytes (16 fp16) along K inside the swizzle
              // atom; MN-major: advance two 8-token groups (2 KB).
              const uint64_t off =
                  static_cast<uint64_t>(TOKMAJOR ? (k * UK * 128) >> 4 : (k * UK * 2) >> 4);
              tc_mma_f16(d_tmem, da + off, db + off, idesc, (kb > c0 || k > 0) ? 1u : 0u);
            }
            tc_commit_multicast(empty_bar(stage), 0x3);  // frees the slot (in both CTAs) when these MMAs finish
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit(accf_bar(acc));  // accumulator ready for the drain warps
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
      }
      // Make sure no MMA is still writing TMEM before it is released.
      tc_commit(drain_bar);
      mbar_wait_bounded(drain_bar, 0, fault);
    }
  } else {
    // ------------------------------------------------------------ drain (8 warps)
    // Warp w reads TMEM lanes 32q..32q+31 (q = w mod 4, the lane quarter it
    // may access) and columns 128h..128h+127 of the tile (h = 0 for warps
    // 2-5, 1 for warps 6-9); each lane sums one row's 128 columns.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    int acc = 0;
    uint32_t acc_phase = 0;
    const int d = s.d;
    bool ok = true;
    for (int job = cid; ok && job < s.jobs; job += nclusters) {
      int ti0, tj, k0, k1;
      job_of(s, job, ti0, tj, k0, k1);
      const int ti = ti0 + rank;
      float sum[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) sum[i] = 0.f;
      for (int c0 = k0; c0 < k1; c0 += CH) {
        if (!mbar_wait_bounded(accf_bar(acc), acc_phase, fault)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v[32];
          tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                 static_cast<uint32_t>(acc * BN + h * 128 + c * 32),
                             v);
#pragma unroll
          for (int i = 0; i < 32; ++i) sum[c * 32 + i] += v[i];
        }
        tc_fence_before();
        mbar_arrive(acce_bar(acc));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) break;
      const int r = ti * BM + q * 32 + lane;
      const int row0 = ti * BM;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int cb = tj * BN + h * 128 + c * 32;
        if (cb + 31 < row0 || cb >= d) continue;  // chunk wholly below the diagonal / outside
        if (r < d) {
          float* srow = S + static_cast<size_t>(r) * d;
          if (cb >= r) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              atomicAdd(reinterpret_cast<float4*>(srow + cb + i),
                        make_float4(sum[c * 32 + i], sum[c * 32 + i + 1], sum[c * 32 + i + 2],
                                    sum[c * 32 + i + 3]));
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (cb + i >= r) atomicAdd(srow + cb + i, sum[c * 32 + i]);
          }
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (cb + i > r) atomicAdd(S + static_cast<size_t>(cb + i) * d + r, sum[c * 32 + i]);
        }
      }
    }
  }

  tc_fence_before();
  cluster_sync();   // neither CTA leaves while the other may still use its shared memory
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

bool make_x_map(CUtensorMap* m, const void* X, int64_t d, int64_t n_tok, int64_t ldx, int box_rows,
                bool tok_major) {
  auto fn = encode_fn();
  if (!fn) return false;
  // channel-major: [d rows][n_tok]; token-major: [n_tok rows][d], box 64 x BK
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(tok_major ? d : n_tok),
                        static_cast<cuuint64_t>(tok_major ? n_tok : d)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldx) * 2};
  cuuint32_t box[2] = {tok_major ? static_cast<cuuint32_t>(TM_BOX) : static_cast<cuuint32_t>(BK),
                       tok_major ? static_cast<cuuint32_t>(BK) : static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(X), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

// Host-side schedule (also used by the tests through gptq_internal_*).
// grid_max: clusters (pairs of CTAs) available.
static SyrkSchedule make_schedule(int64_t d, int64_t n_tok, int grid_max) {
  SyrkSchedule s{};
  s.d = static_cast<int>(d);
  s.kb_total = static_cast<int>((n_tok + BK - 1) / BK);
  s.n_i = static_cast<int>((d + BM - 1) / BM);
  const int n_j = static_cast<int>((d + BN - 1) / BN);
  s.tiles = 0;
  s.pairs = 0;
  for (int j = 0; j < n_j; ++j) {
    const int c = (s.n_i < 2 * j + 2) ? s.n_i : 2 * j + 2;
    s.tiles += c;
    s.pairs += (c + 1) / 2;
  }
  const int G = grid_max;
  s.full = (s.pairs / G) * G;
  s.rem = s.pairs - s.full;
  s.ks = 1;
  if (s.rem > 0) {
    // Pieces of at least 8 slabs; pick the split that best fills the last
    // wave, with a small charge per extra piece for the atomic flushes.
    const int ks_max = std::max(1, std::min(32, s.kb_total / 8));
    double best = 1e30;
    for (int ks = 1; ks <= ks_max; ++ks) {
      const double waves = static_cast<double>((s.rem * ks + G - 1) / G) / ks;
      const double cost = waves + 0.004 * ks;
      if (cost < best - 1e-12) {
        best = cost;
        s.ks = ks;
      }
    }
  }
  s.jobs = s.full + s.rem * s.ks;
  return s;
}

gptq_status_t launch_hessian_syrk(const void* X, int64_t d, int64_t n_tok, int64_t ldx, bool tok_major,
                                  float* S, cudaStream_t st) {
  CUtensorMap tm_a, tm_b;
  if (!make_x_map(&tm_a, X, d, n_tok, ldx, BM, tok_major) ||
      !make_x_map(&tm_b, X, d, n_tok, ldx, BN / 2, tok_major))
    return GPTQ_ERR_CUDA;
  int* fault = fault_word_ptr();
  if (!fault) return GPTQ_ERR_CUDA;
  const int clusters = sm_count() / 2;
  SyrkSchedule s = make_schedule(d, n_tok, clusters);
  auto kern = tok_major ? hessian_syrk_kernel<true> : hessian_syrk_kernel<false>;
  static int attr_dev[2] = {-1, -1};   // the attribute is set once per device and layout
  int dev = 0;
  GPTQ_CUDA_TRY(cudaGetDevice(&dev));
  if (attr_dev[tok_major ? 1 : 0] != dev) {
    GPTQ_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES));
    attr_dev[tok_major ? 1 : 0] = dev;
  }
  // one cluster of two CTAs per pair job in flight
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * std::min(clusters, s.jobs));
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  GPTQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, tm_a, tm_b, s, S, fault));
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

}  // namespace gptq

// Test hook: the schedule the kernel would use (tiles, full jobs, remainder
// tiles, pieces, jobs) for a given problem and grid.
extern "C" GPTQ_API void gptq_internal_syrk_schedule(int64_t d, int64_t n_tok, int grid, int32_t* out5) {
  gptq::SyrkSchedule s = gptq::make_schedule(d, n_tok, grid);
  out5[0] = s.pairs;
  out5[1] = s.full;
  out5[2] = s.rem;
  out5[3] = s.ks;
  out5[4] = s.jobs;
}
