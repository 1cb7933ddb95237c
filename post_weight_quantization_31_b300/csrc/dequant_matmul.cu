// Y = X · Wᵀ with W read from the packed layer and dequantized on the fly:
//   W[n][k] = scales[g][n] * (code[n][k] - zero[g][n]),  g = g_idx[k],
// rounded to X's type (fp16 or bf16), the matmul the GPTQ practical guide
// (m.lqnn.cn/news/117696, §4.3) says a GPTQ layer runs at inference: unpack
// the low-bit codes to 16-bit weights, then multiply.  Here the unpacking
// happens in shared memory right in front of the tensor cores, so HBM only
// carries the packed words.
//
// Tile: 128 output features (n) x MT activation rows (m) per CTA, the MMA
// run as D[n][m] = W_tile · X_tileᵀ (M = 128 n, N = MT m), so that a small
// batch (decode, M = 1..16) still fills an MMA.  K advances in 64-wide slabs.
//   warp 0      TMA: the n-tile's scale table once, then per slab the packed
//               words [2*bits][128 n] and the 64 g_idx entries, into a ring
//               of up to 8 stages that the dequantizers release
//   warp 10     TMA: per slab the X tile [MT x 64] (128-byte swizzle,
//               K-major), into a ring of up to 4 stages that the MMA releases
//   warp 1      MMA issuer: 4 x tcgen05.mma kind::f16 (K = 16) per slab
//   warps 2-9   dequantizers: thread (n, k-half) turns 32 codes of row n into
//               32 16-bit weights, written into the A tile of the operand
//               ring in the 128-byte-swizzle K-major layout (conflict-free
//               16-byte stores); warps 2-5 then read the accumulator from
//               TMEM and write Y.
// The n-tile's scales ([group][n], by TMA) and zero words ([group][4*bits],
// copied by the dequantizers) stay in shared memory for the whole K range
// when they fit (at most 256 groups); otherwise they are read from global
// memory.  With few tiles the K range
// is split over CTAs, which add their partial sums into Y with fp32 atomics
// (Y is cleared first).
#include <algorithm>
#include <type_traits>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace gptq {
namespace {

constexpr int QN = 128;          // output features per CTA
constexpr int QK = 64;           // K per slab (128 bytes of 16-bit values)
constexpr int QUK = 16;          // K of one kind::f16 MMA
constexpr int QTHREADS = 352;    // warp 0 words/table TMA, warp 1 MMA, warps 2-9 dequant, warp 10 X TMA
constexpr int QDQ = 256;         // dequantizing threads
constexpr int QMAXRS = 8;        // packed-word ring depth (at most)
constexpr int QMAXAS = 4;        // operand ring depth (at most)
constexpr size_t QSMEM_MAX = 225 * 1024;

__host__ __device__ constexpr size_t al1k(size_t x) { return (x + 1023) & ~static_cast<size_t>(1023); }

// Shared-memory layout (offsets from a 1024-byte-aligned base):
//   rs x [packed words 2*bits x 128 n | 64 g_idx]   (TMA, released by the dequantizers)
//   as x [A tile 128 n x 64 k | X tile MT x 64 k]   (released by the MMA)
//   scale table [G][128 n] fp32 (TMA), zero words [G][4*bits] (copied), barriers
struct QLayout {
  int rs, as, mt;
  size_t raw, rstage, a, b, astage, sc, zw, bars, total;
  __host__ __device__ QLayout(int bits, int mt_, int n_groups, bool staged, int rs_, int as_) {
    rs = rs_;
    as = as_;
    mt = mt_;
    raw = static_cast<size_t>(2 * bits) * QN * 4;
    rstage = al1k(raw) + 1024;
    a = static_cast<size_t>(QN) * QK * 2;
    b = al1k(static_cast<size_t>(mt) * QK * 2);
    astage = a + b;
    sc = static_cast<size_t>(rs) * rstage + static_cast<size_t>(as) * astage;
    zw = sc + (staged ? al1k(static_cast<size_t>(n_groups) * QN * 4) : 0);
    bars = zw + (staged ? al1k(static_cast<size_t>(n_groups) * 16 * bits) : 0);
    total = bars + 512 + 1024;                             // barriers, TMEM slot, base alignment
  }
  __host__ __device__ size_t raw_off(int s) const { return s * rstage; }
  __host__ __device__ size_t g_off(int s) const { return s * rstage + al1k(raw); }
  __host__ __device__ size_t a_off(int s) const { return rs * rstage + s * astage; }
  __host__ __device__ size_t b_off(int s) const { return rs * rstage + s * astage + a; }
};

struct QArgs {
  int M, N, K, n_groups, n_tiles, m_tiles, ksplit, n_slabs, rs, as, mt;
  float* Y;
  const float* scales;
  const int32_t* qzeros;
};

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Code i of the LSB-first stream w[0], w[1], ... (bits wide).
__device__ __forceinline__ uint32_t stream_code(const int32_t* w, int i, int bits) {
  const int b = i * bits;
  const int k = b >> 5, sh = b & 31;
  uint64_t v = static_cast<uint32_t>(w[k]);
  if (sh + bits > 32) v |= static_cast<uint64_t>(static_cast<uint32_t>(w[k + 1])) << 32;
  return static_cast<uint32_t>((v >> sh) & ((1u << bits) - 1u));
}

// Code c (0..31) of a 32*BITS-bit little-endian stream in wv[], as the float
// 2^23 + code.
template <int BITS>
__device__ __forceinline__ float code_magic(const uint32_t (&wv)[BITS], int c) {
  const int b = c * BITS, k = b >> 5, sh = b & 31;
  uint32_t q = wv[k] >> sh;
  if (sh + BITS > 32) q |= wv[k + 1] << (32 - sh);
  return __uint_as_float(0x4B000000u | (q & ((1u << BITS) - 1u)));
}

__device__ __forceinline__ void fence_proxy_async_smem_q() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void dequant_bar() { asm volatile("bar.sync 1, %0;" ::"n"(QDQ) : "memory"); }

__device__ __forceinline__ int clamp_g(int g, int n_groups) {
  return g < 0 ? 0 : (g >= n_groups ? n_groups - 1 : g);
}

// (a - z) * s for two values at once with the packed fp32x2 instructions
// (each lane rounded to nearest, as the scalar operations would be).
__device__ __forceinline__ float2 sub_mul2(float a0, float a1, float z, float s) {
  unsigned long long x, zz, ss, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(zz) : "f"(z));
  asm("mov.b64 %0, {%1, %1};" : "=l"(ss) : "f"(s));
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(x), "l"(zz));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(d), "l"(ss));
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
  return r;
}

// Bounded wait that sleeps between polls: for the TMA producers, whose
// ring slots free up at slab granularity, so that they leave the issue
// slots to the dequantizing warps.
__device__ __forceinline__ bool mbar_wait_backoff(uint32_t bar, uint32_t parity, int* fault) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*reinterpret_cast<volatile int*>(fault) & kStatTimeout) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        atomicOr(fault, kStatTimeout);
        return false;
      }
    }
  }
}

// Wait by lane 0 (bounded), broadcast the outcome; on success every lane
// also observes the completed phase (its own acquire).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int* fault, int lane) {
  int ok = 1;
  if (lane == 0) ok = mbar_wait_bounded(bar, parity, fault);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) mbar_try_wait(bar, parity);
  return ok != 0;
}

template <typename T, int BITS, bool STAGED>
__global__ void __launch_bounds__(QTHREADS, 2)
    dqgemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_s, QArgs p,
                  int* fault) {
  extern __shared__ uint8_t q_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(q_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int RS = p.rs, AS = p.as, mt = p.mt;
  const QLayout L(BITS, mt, p.n_groups, STAGED, RS, AS);
  const uint32_t bar0 = smem_u32(sm + L.bars);
  auto raw_full = [&](int i) { return bar0 + 8u * i; };                   // TMA: words + g_idx
  auto raw_empty = [&](int i) { return bar0 + 8u * (QMAXRS + i); };       // dequantizers done
  auto x_full = [&](int i) { return bar0 + 8u * (2 * QMAXRS + i); };      // TMA: X tile
  auto a_full = [&](int i) { return bar0 + 8u * (2 * QMAXRS + QMAXAS + i); };   // A tile written
  auto ab_empty = [&](int i) { return bar0 + 8u * (2 * QMAXRS + 2 * QMAXAS + i); };  // MMA done
  const uint32_t tab_bar = bar0 + 8u * (2 * QMAXRS + 3 * QMAXAS);
  const uint32_t acc_bar = tab_bar + 8u;
  const uint32_t drain_bar = tab_bar + 16u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L.bars + 8 * (2 * QMAXRS + 3 * QMAXAS + 3));
  const float* sc_t = reinterpret_cast<const float*>(sm + L.sc);
  uint32_t* zw_t = reinterpret_cast<uint32_t*>(sm + L.zw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ks = blockIdx.x % p.ksplit;
  const int tile = blockIdx.x / p.ksplit;
  const int nt = tile % p.n_tiles, mtile = tile / p.n_tiles;
  const int n0 = nt * QN, m0 = mtile * mt;
  const int sl0 = static_cast<int>(static_cast<long long>(p.n_slabs) * ks / p.ksplit);
  const int sl1 = static_cast<int>(static_cast<long long>(p.n_slabs) * (ks + 1) / p.ksplit);
  const int nsl = sl1 - sl0;
  uint32_t tmem_cols = 32;
  while (tmem_cols < static_cast<uint32_t>(mt)) tmem_cols <<= 1;
  const int zrow = 4 * BITS;             // zero words of one group for the tile's 128 rows

  if (threadIdx.x == 0) {
    for (int i = 0; i < RS; ++i) {
      mbar_init(raw_full(i), 1);
      mbar_init(raw_empty(i), QDQ / 32);
    }
    for (int i = 0; i < AS; ++i) {
      mbar_init(x_full(i), 1);
      mbar_init(a_full(i), QDQ / 32);
      mbar_init(ab_empty(i), 1);
    }
    mbar_init(tab_bar, 1);
    mbar_init(acc_bar, 1);
    mbar_init(drain_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------- packed words, g_idx, scale table
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_g);
      if constexpr (STAGED) {
        tma_prefetch_desc(&tm_s);
        mbar_arrive_expect_tx(tab_bar, static_cast<uint32_t>(p.n_groups) * QN * 4);
        for (int g0 = 0; g0 < p.n_groups; g0 += 256)
          tma_load_2d(smem_u32(sm + L.sc) + g0 * QN * 4, &tm_s, tab_bar, n0, g0);
      }
      const uint32_t tx = static_cast<uint32_t>(L.raw + QK * 4);
      int s = 0;
      uint32_t ph = 0;
      for (int i = 0; i < nsl; ++i) {
        if (i >= RS && !mbar_wait_backoff(raw_empty(s), ph ^ 1u, fault)) break;
        const int k0 = (sl0 + i) * QK;
        mbar_arrive_expect_tx(raw_full(s), tx);
        tma_load_2d(smem_u32(sm + L.raw_off(s)), &tm_q, raw_full(s), n0, k0 * BITS / 32);
        tma_load_2d(smem_u32(sm + L.g_off(s)), &tm_g, raw_full(s), k0, 0);
        if (++s == RS) { s = 0; ph ^= 1u; }
      }
    }
  } else if (warp == QTHREADS / 32 - 1) {
    // ------------------------------------------- activation tiles
    if (lane == 0) {
      tma_prefetch_desc(&tm_x);
      const uint32_t tx = static_cast<uint32_t>(mt) * QK * 2;
      int s = 0;
      uint32_t ph = 0;
      for (int i = 0; i < nsl; ++i) {
        if (i >= AS && !mbar_wait_backoff(ab_empty(s), ph ^ 1u, fault)) break;
        mbar_arrive_expect_tx(x_full(s), tx);
        tma_load_2d(smem_u32(sm + L.b_off(s)), &tm_x, x_full(s), (sl0 + i) * QK, m0);
        if (++s == AS) { s = 0; ph ^= 1u; }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr int fmt = std::is_same<T, __nv_bfloat16>::value ? 1 : 0;   // 0 = f16, 1 = bf16
      const uint32_t idesc = make_idesc(QN, mt, fmt, fmt);
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int i = 0; i < nsl && ok; ++i) {
        ok = mbar_wait_bounded(x_full(s), ph, fault) && mbar_wait_bounded(a_full(s), ph, fault);
        if (!ok) break;
        tc_fence_after();
        const uint64_t da = smem_desc_sw128_kmajor(smem_u32(sm + L.a_off(s)));
        const uint64_t db = smem_desc_sw128_kmajor(smem_u32(sm + L.b_off(s)));
#pragma unroll
        for (int k = 0; k < QK / QUK; ++k) {
          const uint64_t off = static_cast<uint64_t>((k * QUK * 2) >> 4);   // 32 bytes per step
          tc_mma_f16(tmem_base, da + off, db + off, idesc, (i == 0 && k == 0) ? 0u : 1u);
        }
        tc_commit(ab_empty(s));
        if (++s == AS) { s = 0; ph ^= 1u; }
      }
      if (ok) tc_commit(acc_bar);
      tc_commit(drain_bar);
      mbar_wait_bounded(drain_bar, 0, fault);
    }
  } else {
    // ------------------------------------------- dequantizers (warps 2-9)
    const int t = threadIdx.x - 64;
    const int nn = t & (QN - 1), half = t >> 7;    // row of the tile, k-half of the slab
    const int n = n0 + nn;
    bool ok = true;
    // this row's zero-point: bits [nn*BITS, (nn+1)*BITS) of a group's zero words
    const int zk = (nn * BITS) >> 5, zsh = (nn * BITS) & 31;
    const bool zstr = zsh + BITS > 32;
    if constexpr (STAGED) {
      // the tile's zero words for every group, 4*BITS per group
      const int zstride = p.N * BITS / 32;
      const int total = p.n_groups * zrow;
#pragma unroll 4
      for (int i = t; i < total; i += QDQ) {
        const int g = i / zrow, w = i % zrow;
        const int col = n0 * BITS / 32 + w;
        zw_t[i] = col < zstride ? static_cast<uint32_t>(__ldg(p.qzeros + static_cast<size_t>(g) * zstride + col)) : 0u;
      }
      dequant_bar();
      ok = warp_wait(tab_bar, 0, fault, lane);
    }
    auto zero_of = [&](int g) -> uint32_t {
      if constexpr (STAGED) {
        const uint32_t* zr = zw_t + g * zrow;
        uint32_t v = zr[zk] >> zsh;
        if (zstr) v |= zr[zk + 1] << (32 - zsh);
        return v & ((1u << BITS) - 1u);
      } else {
        return n < p.N ? stream_code(p.qzeros + static_cast<size_t>(g) * (p.N * BITS / 32), n, BITS) : 0u;
      }
    };
    auto scale_of = [&](int g) -> float {
      if constexpr (STAGED) return sc_t[g * QN + nn];
      else return n < p.N ? __ldg(p.scales + static_cast<size_t>(g) * p.N + n) : 0.f;
    };
    int rs = 0, as = 0;
    uint32_t rph = 0, aph = 0;
    for (int i = 0; i < nsl && ok; ++i) {
      if (!warp_wait(raw_full(rs), rph, fault, lane)) { ok = false; break; }
      const uint32_t* raw = reinterpret_cast<const uint32_t*>(sm + L.raw_off(rs));
      const int* gsl = reinterpret_cast<const int*>(sm + L.g_off(rs)) + 32 * half;
      uint32_t wv[BITS];
#pragma unroll
      for (int b = 0; b < BITS; ++b) wv[b] = raw[(half * BITS + b) * QN + nn];
      if (i >= AS && !warp_wait(ab_empty(as), aph ^ 1u, fault, lane)) { ok = false; break; }
      const uint32_t arow = smem_u32(sm + L.a_off(as)) + nn * 128;
      // One group for the whole slab (no act-order, group size >= 64): one
      // scale/zero lookup for all 32 weights.
      const int* gslab = reinterpret_cast<const int*>(sm + L.g_off(rs));
      const int2 gpair = *reinterpret_cast<const int2*>(gslab + 2 * lane);
      const int gfirst = __shfl_sync(0xffffffffu, gpair.x, 0);
      if (__all_sync(0xffffffffu, gpair.x == gfirst && gpair.y == gfirst)) {
        const int g = clamp_g(gfirst, p.n_groups);
        const float sv = scale_of(g);
        const float zv = __uint_as_float(0x4B000000u | zero_of(g));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t xv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 r = sub_mul2(code_magic<BITS>(wv, 8 * j + 2 * e), code_magic<BITS>(wv, 8 * j + 2 * e + 1),
                                      zv, sv);
            xv[e] = pack2<T>(r.x, r.y);
          }
          const uint32_t x0 = xv[0], x1 = xv[1], x2 = xv[2], x3 = xv[3];
          const int chunk = 4 * half + j;
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(arow + 16 * (chunk ^ (nn & 7))),
                       "r"(x0), "r"(x1), "r"(x2), "r"(x3)
                       : "memory");
        }
      } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {                // 8 weights = one 16-byte chunk
        const int4 ga = *reinterpret_cast<const int4*>(gsl + 8 * j);
        const int4 gb = *reinterpret_cast<const int4*>(gsl + 8 * j + 4);
        const bool uni = ga.x == ga.y && ga.x == ga.z && ga.x == ga.w && ga.x == gb.x && ga.x == gb.y &&
                         ga.x == gb.z && ga.x == gb.w;
        float v[8];
        if (uni) {
          const int g = clamp_g(ga.x, p.n_groups);
          const float sv = scale_of(g);
          const float zv = __uint_as_float(0x4B000000u | zero_of(g));
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = sv * (code_magic<BITS>(wv, 8 * j + e) - zv);
        } else {
          const int gv[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int g = clamp_g(gv[e], p.n_groups);
            v[e] = scale_of(g) * (code_magic<BITS>(wv, 8 * j + e) -
                                  __uint_as_float(0x4B000000u | zero_of(g)));
          }
        }
        const uint32_t x0 = pack2<T>(v[0], v[1]), x1 = pack2<T>(v[2], v[3]);
        const uint32_t x2 = pack2<T>(v[4], v[5]), x3 = pack2<T>(v[6], v[7]);
        const int chunk = 4 * half + j;           // logical 16-byte chunk of the 128-byte row
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(arow + 16 * (chunk ^ (nn & 7))),
                     "r"(x0), "r"(x1), "r"(x2), "r"(x3)
                     : "memory");
      }
      }
      fence_proxy_async_smem_q();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(a_full(as));
        mbar_arrive(raw_empty(rs));
      }
      if (++rs == RS) { rs = 0; rph ^= 1u; }
      if (++as == AS) { as = 0; aph ^= 1u; }
    }
    // ------------------------------------------- epilogue (warps 2-5)
    if (ok && warp < 6 && nsl > 0) {
      const int q = warp & 3;                     // TMEM lane quarter this warp may read
      const int nrow = n0 + 32 * q + lane;
      if (warp_wait(acc_bar, 0, fault, lane)) {
        tc_fence_after();
        for (int c0 = 0; c0 < mt; c0 += 32) {
          float v[32];
          tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c0), v);
          if (nrow < p.N) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int m = m0 + c0 + e;
              if (c0 + e < mt && m < p.M) {
                float* dst = p.Y + static_cast<size_t>(m) * p.N + nrow;
                if (p.ksplit > 1) atomicAdd(dst, v[e]);
                else *dst = v[e];
              }
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

template <typename T, int BITS, bool STAGED>
gptq_status_t launch_q(const CUtensorMap& tx, const CUtensorMap& tq, const CUtensorMap& tg, const CUtensorMap& ts,
                       QArgs p, cudaStream_t st) {
  const QLayout L(BITS, p.mt, p.n_groups, STAGED, p.rs, p.as);
  auto kern = dqgemm_kernel<T, BITS, STAGED>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L.total)) !=
      cudaSuccess)
    return GPTQ_ERR_CUDA;
  // Split K so that the grid fills the SMs (one CTA per SM), keeping at
  // least 4 slabs per CTA for the pipeline.
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, QTHREADS, L.total) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int slots = sm_count() * per_sm;
  // Split K over CTAs when Y is small (the partial sums go through fp32
  // atomics into a cleared Y): pick the split whose busiest SM has the
  // fewest slabs to do (CTAs per SM x slabs per CTA, plus about two slabs
  // of start-up per CTA).
  const int sms = sm_count();
  const int tiles = p.n_tiles * p.m_tiles;
  int ks = 1;
  if (static_cast<long long>(p.M) * p.N <= (4ll << 20)) {
    long long best = -1;
    for (int k = 1; k <= std::max(1, p.n_slabs / 4); ++k) {
      const long long per_sm = (static_cast<long long>(tiles) * k + sms - 1) / sms;
      const long long cost = per_sm * ((p.n_slabs + k - 1) / k + 2);
      if (best < 0 || cost < best) {
        best = cost;
        ks = k;
      }
    }
  }
  (void)slots;
  p.ksplit = ks;
  if (ks > 1 && cudaMemsetAsync(p.Y, 0, sizeof(float) * static_cast<size_t>(p.M) * p.N, st) != cudaSuccess)
    return GPTQ_ERR_CUDA;
  kern<<<tiles * ks, QTHREADS, L.total, st>>>(tx, tq, tg, ts, p, fault_word_ptr());
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

// Ring depths: the scale/zero table staged if possible; for small MT
// (decode) the smallest rings that still pipeline (4 word stages, 2 operand
// stages) so that two CTAs share an SM, else the deepest rings that fit.
template <typename T, int BITS>
gptq_status_t launch_bits_q(const CUtensorMap& tx, const CUtensorMap& tq, const CUtensorMap& tg,
                            const CUtensorMap& ts, QArgs p, cudaStream_t st) {
  // The scale table arrives as one TMA box, so at most 256 groups are staged.
  for (int staged = p.n_groups <= 256 ? 1 : 0; staged >= 0; --staged) {
    if (p.mt <= 64 && QLayout(BITS, p.mt, p.n_groups, staged != 0, 4, 2).total <= QSMEM_MAX / 2) {
      p.rs = 4;
      p.as = 2;
      return staged ? launch_q<T, BITS, true>(tx, tq, tg, ts, p, st)
                    : launch_q<T, BITS, false>(tx, tq, tg, ts, p, st);
    }
    for (int as = QMAXAS; as >= 2; --as)
      for (int rs = QMAXRS; rs >= 2; rs -= 2)
        if (QLayout(BITS, p.mt, p.n_groups, staged != 0, rs, as).total <= QSMEM_MAX) {
          p.rs = rs;
          p.as = as;
          return staged ? launch_q<T, BITS, true>(tx, tq, tg, ts, p, st)
                        : launch_q<T, BITS, false>(tx, tq, tg, ts, p, st);
        }
  }
  return GPTQ_ERR_UNSUPPORTED;
}

template <typename T>
gptq_status_t launch_dt_q(const CUtensorMap& tx, const CUtensorMap& tq, const CUtensorMap& tg, const CUtensorMap& ts,
                          QArgs p, int bits, cudaStream_t st) {
  switch (bits) {
    case 2: return launch_bits_q<T, 2>(tx, tq, tg, ts, p, st);
    case 3: return launch_bits_q<T, 3>(tx, tq, tg, ts, p, st);
    case 4: return launch_bits_q<T, 4>(tx, tq, tg, ts, p, st);
    default: return launch_bits_q<T, 8>(tx, tq, tg, ts, p, st);
  }
}

}  // namespace

gptq_status_t launch_dequant_matmul(const void* X, int x_dtype, int64_t M, int64_t ldx, const int32_t* qweight,
                                    const int32_t* qzeros, const float* scales, const int32_t* g_idx,
                                    int64_t d_row, int64_t d_col, int bits, int n_groups, float* Y,
                                    cudaStream_t st) {
  auto fn = encode_fn();
  if (!fn || !fault_word_ptr()) return GPTQ_ERR_CUDA;
  const int mt = static_cast<int>(std::min<int64_t>(256, (M + 15) / 16 * 16));
  CUtensorMap tx, tq, tg;
  {  // X [M][K] 16-bit, box 64 K x MT rows, 128-byte swizzle
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(d_col), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldx) * 2};
    cuuint32_t box[2] = {QK, static_cast<cuuint32_t>(mt)};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&tx, x_dtype == GPTQ_W_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
           const_cast<void*>(X), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return GPTQ_ERR_INVALID_ARG;
  }
  {  // qweight [K*bits/32][N] int32, box 128 n x 2*bits words
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(d_row), static_cast<cuuint64_t>(d_col * bits / 32)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(d_row) * 4};
    cuuint32_t box[2] = {QN, static_cast<cuuint32_t>(2 * bits)};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&tq, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<int32_t*>(qweight), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return GPTQ_ERR_INVALID_ARG;
  }
  {  // g_idx [K] int32 as one row, box 64
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(d_col), 1};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(d_col) * 4};
    cuuint32_t box[2] = {QK, 1};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&tg, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<int32_t*>(g_idx), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return GPTQ_ERR_INVALID_ARG;
  }
  CUtensorMap ts;
  {  // scales [G][N] fp32, box 128 n x min(G, 256) groups
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(d_row), static_cast<cuuint64_t>(n_groups)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(d_row) * 4};
    cuuint32_t box[2] = {QN, static_cast<cuuint32_t>(std::min(n_groups, 256))};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(scales), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return GPTQ_ERR_INVALID_ARG;
  }
  QArgs p{};
  p.mt = mt;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(d_row);
  p.K = static_cast<int>(d_col);
  p.n_groups = n_groups;
  p.n_tiles = static_cast<int>((d_row + QN - 1) / QN);
  p.m_tiles = static_cast<int>((M + mt - 1) / mt);
  p.n_slabs = static_cast<int>(d_col / QK);
  p.ksplit = 1;
  p.Y = Y;
  p.scales = scales;
  p.qzeros = qzeros;
  if (x_dtype == GPTQ_W_BF16) return launch_dt_q<__nv_bfloat16>(tx, tq, tg, ts, p, bits, st);
  return launch_dt_q<__half>(tx, tq, tg, ts, p, bits, st);
}

}  // namespace gptq
