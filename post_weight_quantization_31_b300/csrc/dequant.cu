// The packed layer back to dense weights:
//   W[r][c] = scales[g][r] * (code[r][c] - zero[g][r]),  g = g_idx[c],
// in the original column order.  With act-order the columns of one group are
// scattered over the row, and g_idx maps each column to its group: the
// re-ordering the GPTQ practical guide (m.lqnn.cn/news/117696, §5.2) says
// happens when a desc_act model is loaded.  The packed layouts are those of
// gptq_pack (pack.cu).
//
// The work is HBM-bound: per weight, bits/8 bytes of codes in and 2 (or 4)
// bytes out.  The layer is cut into tiles of 32 rows x 256 columns; a
// persistent grid (one wave of resident CTAs) gives each CTA an equal run of
// consecutive tiles, row block by row block.
//   * A producer thread streams each tile's qweight words and its 256 g_idx
//     entries into a 4-stage shared-memory ring with TMA (words: box 32 rows
//     (inner) x 8*bits words, so a tile arrives as [word][row]); the compute
//     warps issue no global loads per tile.
//   * Eight compute warps each own 32 columns of the tile; lane = row.  A
//     warp's 32 columns are exactly `bits` words of every row, so each lane
//     reads `bits` consecutive-row words (no bank conflicts) and holds its
//     row's 32 codes in registers.
//   * The 32 rows' scales and zero-points of every group are staged once per
//     row block in shared memory as [group][row], so the lanes of a warp
//     read 32 consecutive words whatever the group (act-order included).
//     When a warp's 32 columns all fall in one group (no act-order), the
//     pair is read once.
//   * Each warp writes its 32 x 32 result into its own swizzled shared tile
//     (conflict-free 16-byte stores, one row per lane) and sends it to HBM
//     with a TMA store; two tiles per warp alternate so that the store of
//     one overlaps the computation of the next.
// Layers whose scale table does not fit in shared memory (more than about
// 700 groups) read scales and zeros from global memory instead (coalesced:
// lane = row).
//
// Exactness: code - zero is a small integer; it is formed exactly as
// (2^23 + code) - (2^23 + zero) in fp32, multiplied by the scale once and
// rounded once to the output type, as the formula reads.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace gptq {
namespace {

constexpr int DQ_RB = 32;                        // rows per tile (= lanes)
constexpr int DQ_CHUNK = 256;                    // columns per tile
constexpr int DQ_CWARPS = DQ_CHUNK / 32;         // compute warps, 32 columns each
constexpr int DQ_THREADS = (DQ_CWARPS + 1) * 32; // + one producer warp
constexpr int DQ_STAGES = 4;
constexpr size_t DQ_SMEM_LIMIT = 200 * 1024;

__host__ __device__ constexpr size_t align1k(size_t x) { return (x + 1023) & ~static_cast<size_t>(1023); }

// Shared-memory layout (offsets from a 1024-byte-aligned base).
struct DqLayout {
  size_t stage_bytes, words, out, sc, z, total;
  __host__ __device__ DqLayout(int bits, int out_bytes, int n_groups, bool staged) {
    // 8*bits words x 32 rows, then the tile's 256 g_idx entries
    stage_bytes = static_cast<size_t>(8 * bits) * DQ_RB * 4 + DQ_CHUNK * 4;
    words = 1024;                                                  // after the mbarriers
    out = words + DQ_STAGES * stage_bytes;
    const size_t out_tile = static_cast<size_t>(32) * 32 * out_bytes;
    sc = out + static_cast<size_t>(DQ_CWARPS) * 2 * out_tile;
    z = sc + (staged ? static_cast<size_t>(n_groups) * 32 * 4 : 0);
    total = align1k(z + (staged ? static_cast<size_t>(n_groups) * 32 : 0)) + 1024;  // + base alignment
  }
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

// Code c (0..31) of a row's 32*BITS-bit little-endian stream held in wv[],
// as the float 2^23 + code.
template <int BITS>
__device__ __forceinline__ float code_magic(const uint32_t (&wv)[BITS], int c) {
  const int b = c * BITS, k = b >> 5, sh = b & 31;
  uint32_t q = wv[k] >> sh;
  if (sh + BITS > 32) q |= wv[k + 1] << (32 - sh);
  return __uint_as_float(0x4B000000u | (q & ((1u << BITS) - 1u)));
}

__device__ __forceinline__ void tma_store_2d(const void* tmap, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_le1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void compute_bar() { asm volatile("bar.sync 1, %0;" ::"n"(DQ_CWARPS * 32) : "memory"); }

// One warp's 32 x 32 output tile (lane = row r, 32 codes in wv) into its
// swizzled shared tile at `ob`: 64-byte rows with the 64B pattern for 2-byte
// outputs, 128-byte rows with the 128B pattern for 4-byte outputs.
// MODE 0: all 32 columns in one group (scale s_u, 2^23 + zero z_u);
// MODE 1: per-column group from the staged [group][row] table;
// MODE 2: per-column group read from global memory.
template <typename T, int BITS, int MODE>
__device__ __forceinline__ void emit_tile(const uint32_t (&wv)[BITS], int gl, float s_u, float z_u,
                                          const float* sc_s, const uint8_t* z_s,
                                          const float* __restrict__ scales,
                                          const int32_t* __restrict__ qzeros, int d_row, int zwords,
                                          int r, int lane, uint32_t ob) {
  constexpr int EPC = 16 / sizeof(T);          // outputs per 16-byte chunk
#pragma unroll
  for (int cc = 0; cc < 32 / EPC; ++cc) {
    float v[EPC];
#pragma unroll
    for (int e = 0; e < EPC; ++e) {
      const int c = cc * EPC + e;
      float sv = s_u, zv = z_u;
      if constexpr (MODE == 1) {
        const int g = __shfl_sync(0xffffffffu, gl, c);
        sv = sc_s[g * 32 + lane];
        zv = __uint_as_float(0x4B000000u | z_s[g * 32 + lane]);
      } else if constexpr (MODE == 2) {
        const int g = __shfl_sync(0xffffffffu, gl, c);
        sv = __ldg(scales + static_cast<size_t>(g) * d_row + r);
        zv = __uint_as_float(0x4B000000u |
                             stream_code(qzeros + static_cast<size_t>(g) * zwords, r, BITS));
      }
      v[e] = sv * (code_magic<BITS>(wv, c) - zv);
    }
    uint4 pk;
    if constexpr (sizeof(T) == 4) {
      pk = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                      __float_as_uint(v[3]));
    } else {
      pk = make_uint4(pack2<T>(v[0], v[1]), pack2<T>(v[2], v[3]), pack2<T>(v[4], v[5]),
                      pack2<T>(v[6], v[7]));
    }
    uint32_t off;
    if constexpr (sizeof(T) == 4) off = lane * 128 + 16 * (cc ^ (lane & 7));
    else off = lane * 64 + 16 * (cc ^ ((lane >> 1) & 3));
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(ob + off), "r"(pk.x), "r"(pk.y),
                 "r"(pk.z), "r"(pk.w)
                 : "memory");
  }
}

template <typename T, int BITS, bool STAGED>
__global__ void __launch_bounds__(DQ_THREADS, 4) dequant_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_w,
    const int32_t* __restrict__ qzeros, const float* __restrict__ scales,
    const __grid_constant__ CUtensorMap tm_g, int d_row, int d_col, int n_groups, int* fault,
    int stall, unsigned long long wait_ns) {
  extern __shared__ unsigned char dq_raw[];
  const uint32_t raw = smem_u32(dq_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = dq_raw + (base - raw);
  const DqLayout L(BITS, sizeof(T), n_groups, STAGED);
  const uint32_t bar_full = base, bar_empty = base + 8 * DQ_STAGES;
  const uint32_t* words = reinterpret_cast<const uint32_t*>(gbase + L.words);
  float* sc_s = reinterpret_cast<float*>(gbase + L.sc);
  uint8_t* z_s = reinterpret_cast<uint8_t*>(gbase + L.z);
  const int words_per_stage = 8 * BITS * DQ_RB;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_chunks = (d_col + DQ_CHUNK - 1) / DQ_CHUNK;
  const long long tiles = static_cast<long long>(d_row / DQ_RB) * n_chunks;
  const long long t0 = tiles * blockIdx.x / gridDim.x, t1 = tiles * (blockIdx.x + 1) / gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < DQ_STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, DQ_CWARPS);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == DQ_CWARPS) {
    // ---------------------------------------------------------------- producer
    if (lane != 0) return;
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_g);
    const uint32_t stage_bytes = static_cast<uint32_t>(L.stage_bytes);
    long long issued = 0;
    int rb = static_cast<int>(t0 / n_chunks), ch = static_cast<int>(t0 % n_chunks);
    int s = 0;
    uint32_t ph = 0;                              // parity of the ring's current pass
    // `stall` (a test launch only): issue no copy at all, so that every wait
    // of the compute warps runs out while nothing is in flight.
    for (long long t = t0; !stall && t < t1; ++t) {
      if (issued >= DQ_STAGES && !mbar_wait_bounded(bar_empty + 8 * s, ph ^ 1u, fault, wait_ns)) break;
      mbar_arrive_expect_tx(bar_full + 8 * s, stage_bytes);
      const uint32_t dst = base + static_cast<uint32_t>(L.words + s * L.stage_bytes);
      tma_load_2d(dst, &tm_q, bar_full + 8 * s, rb * DQ_RB, ch * DQ_CHUNK * BITS / 32);
      tma_load_2d(dst + 4 * (8 * BITS * DQ_RB), &tm_g, bar_full + 8 * s, ch * DQ_CHUNK, 0);
      ++issued;
      if (++ch == n_chunks) { ch = 0; ++rb; }
      if (++s == DQ_STAGES) { s = 0; ph ^= 1u; }
    }
    // Do not leave with copies in flight: wait (bounded) for the last loads.
    for (long long i = issued - DQ_STAGES < 0 ? 0 : issued - DQ_STAGES; i < issued; ++i)
      mbar_wait_bounded(bar_full + 8 * static_cast<int>(i % DQ_STAGES),
                        static_cast<uint32_t>((i / DQ_STAGES) & 1), fault, wait_ns);
    return;
  }

  // ------------------------------------------------------------------ compute
  tma_prefetch_desc(&tm_w);
  const int zwords = d_row * BITS / 32;   // words per group row of qzeros
  const uint32_t out0 = base + static_cast<uint32_t>(L.out) + warp * 2 * (32 * 32 * sizeof(T));
  int cur_rb = -1;
  bool ok = true;
  int n_stores = 0;
  int rb = static_cast<int>(t0 / n_chunks), ch = static_cast<int>(t0 % n_chunks);
  int s = 0;
  uint32_t ph = 0;
  for (long long t = t0; t < t1; ++t) {
    const int r0 = rb * DQ_RB;
    if constexpr (STAGED) {
      if (rb != cur_rb) {       // every compute warp takes this branch at the same tile
        compute_bar();
        for (int idx = warp * 32 + lane; idx < n_groups * 32; idx += DQ_CWARPS * 32) {
          const int g = idx >> 5, rr = idx & 31;
          sc_s[idx] = __ldg(scales + static_cast<size_t>(g) * d_row + r0 + rr);
          z_s[idx] = static_cast<uint8_t>(stream_code(qzeros + static_cast<size_t>(g) * zwords, r0 + rr, BITS));
        }
        compute_bar();
        cur_rb = rb;
      }
    }
    int w_ok = 1;
    if (lane == 0 && ok) w_ok = mbar_wait_bounded(bar_full + 8 * s, ph, fault, wait_ns);
    ok = ok && __shfl_sync(0xffffffffu, w_ok, 0);
    const int c0 = ch * DQ_CHUNK + warp * 32;     // this warp's first column
    const bool active = ok && c0 < d_col;         // d_col is a multiple of 32
    const int s_cur = s;
    if (ok) mbar_try_wait(bar_full + 8 * s, ph);   // completed: gives every lane the acquire
    if (++ch == n_chunks) { ch = 0; ++rb; }
    if (++s == DQ_STAGES) { s = 0; ph ^= 1u; }
    uint32_t wv[BITS];
    int gl = 0;
    if (active) {
      const uint32_t* ws = words + s_cur * (L.stage_bytes / 4);
#pragma unroll
      for (int b = 0; b < BITS; ++b) wv[b] = ws[(warp * BITS + b) * 32 + lane];
      gl = static_cast<int>(ws[words_per_stage + warp * 32 + lane]);
      gl = gl < 0 ? 0 : (gl >= n_groups ? n_groups - 1 : gl);   // keeps bad input in bounds
    }
    __syncwarp();
    if (lane == 0 && ok) mbar_arrive(bar_empty + 8 * s_cur);
    if (!active) continue;

    // this warp's output tile: wait until the store that last used it has read it
    const uint32_t ob = out0 + (n_stores & 1) * (32 * 32 * sizeof(T));
    if (lane == 0 && n_stores >= 2) bulk_wait_read_le1();
    __syncwarp();

    const int r = r0 + lane;
    const int g0 = __shfl_sync(0xffffffffu, gl, 0);
    const bool uni = __all_sync(0xffffffffu, gl == g0);
    if (uni) {
      float s_u, z_u;
      if constexpr (STAGED) {
        s_u = sc_s[g0 * 32 + lane];
        z_u = __uint_as_float(0x4B000000u | z_s[g0 * 32 + lane]);
      } else {
        s_u = __ldg(scales + static_cast<size_t>(g0) * d_row + r);
        z_u = __uint_as_float(0x4B000000u | stream_code(qzeros + static_cast<size_t>(g0) * zwords, r, BITS));
      }
      emit_tile<T, BITS, 0>(wv, gl, s_u, z_u, sc_s, z_s, scales, qzeros, d_row, zwords, r, lane, ob);
    } else {
      emit_tile<T, BITS, STAGED ? 1 : 2>(wv, gl, 0.f, 0.f, sc_s, z_s, scales, qzeros, d_row, zwords, r,
                                         lane, ob);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(&tm_w, ob, c0, r0);
      bulk_commit();
    }
    ++n_stores;
  }
  if (lane == 0) bulk_wait_all();
  __syncwarp();
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

template <typename T, int BITS, bool STAGED>
gptq_status_t launch_t(const CUtensorMap& tq, const CUtensorMap& tw, const CUtensorMap& tg,
                       const int32_t* qzeros, const float* scales, int d_row, int d_col, int n_groups,
                       cudaStream_t st, int stall, unsigned long long wait_ns) {
  const DqLayout L(BITS, sizeof(T), n_groups, STAGED);
  auto kern = dequant_kernel<T, BITS, STAGED>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L.total)) !=
      cudaSuccess)
    return GPTQ_ERR_CUDA;
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, DQ_THREADS, L.total) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const long long tiles = static_cast<long long>(d_row / DQ_RB) * ((d_col + DQ_CHUNK - 1) / DQ_CHUNK);
  const long long slots = static_cast<long long>(sm_count()) * per_sm;
  const unsigned grid = static_cast<unsigned>(tiles < slots ? tiles : slots);
  kern<<<grid, DQ_THREADS, L.total, st>>>(tq, tw, qzeros, scales, tg, d_row, d_col, n_groups,
                                         fault_word_ptr(), stall, wait_ns);
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

template <typename T, int BITS>
gptq_status_t launch_bits(const CUtensorMap& tq, const CUtensorMap& tw, const CUtensorMap& tg,
                          const int32_t* qzeros, const float* scales, int d_row, int d_col, int n_groups,
                          cudaStream_t st, int stall, unsigned long long wait_ns) {
  if (DqLayout(BITS, sizeof(T), n_groups, true).total <= DQ_SMEM_LIMIT)
    return launch_t<T, BITS, true>(tq, tw, tg, qzeros, scales, d_row, d_col, n_groups, st, stall, wait_ns);
  return launch_t<T, BITS, false>(tq, tw, tg, qzeros, scales, d_row, d_col, n_groups, st, stall, wait_ns);
}

template <typename T>
gptq_status_t launch_dt(const CUtensorMap& tq, const CUtensorMap& tw, const CUtensorMap& tg,
                        const int32_t* qzeros, const float* scales, int d_row, int d_col, int bits,
                        int n_groups, cudaStream_t st, int stall, unsigned long long wait_ns) {
  switch (bits) {
    case 2: return launch_bits<T, 2>(tq, tw, tg, qzeros, scales, d_row, d_col, n_groups, st, stall, wait_ns);
    case 3: return launch_bits<T, 3>(tq, tw, tg, qzeros, scales, d_row, d_col, n_groups, st, stall, wait_ns);
    case 4: return launch_bits<T, 4>(tq, tw, tg, qzeros, scales, d_row, d_col, n_groups, st, stall, wait_ns);
    default: return launch_bits<T, 8>(tq, tw, tg, qzeros, scales, d_row, d_col, n_groups, st, stall, wait_ns);
  }
}

}  // namespace

gptq_status_t launch_dequant_impl(const int32_t* qweight, const int32_t* qzeros, const float* scales,
                                  const int32_t* g_idx, int64_t d_row, int64_t d_col, int bits,
                                  int n_groups, int out_dtype, void* W, cudaStream_t st, int stall,
                                  unsigned long long wait_ns) {
  auto fn = encode_fn();
  if (!fn || !fault_word_ptr()) return GPTQ_ERR_CUDA;
  const int out_bytes = out_dtype == GPTQ_W_FP32 ? 4 : 2;
  // qweight [d_col*bits/32][d_row] int32: box 32 rows x 8*bits words
  CUtensorMap tq, tw;
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(d_row), static_cast<cuuint64_t>(d_col * bits / 32)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(d_row) * 4};
    cuuint32_t box[2] = {DQ_RB, static_cast<cuuint32_t>(8 * bits)};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&tq, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<int32_t*>(qweight), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return GPTQ_ERR_INVALID_ARG;
  }
  // W [d_row][d_col]: box 32 columns x 32 rows, swizzled as the kernel writes it
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(d_col), static_cast<cuuint64_t>(d_row)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(d_col) * out_bytes};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&tw, out_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, W, dims,
           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           out_bytes == 4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return GPTQ_ERR_INVALID_ARG;
  }
  // g_idx [d_col] int32 as a one-row 2-D tensor: box 256 entries (the tail is zero-filled)
  CUtensorMap tg;
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(d_col), 1};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(d_col) * 4};
    cuuint32_t box[2] = {DQ_CHUNK, 1};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&tg, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<int32_t*>(g_idx), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return GPTQ_ERR_INVALID_ARG;
  }
  const int r = static_cast<int>(d_row), c = static_cast<int>(d_col);
  if (out_dtype == GPTQ_W_FP32)
    return launch_dt<float>(tq, tw, tg, qzeros, scales, r, c, bits, n_groups, st, stall, wait_ns);
  if (out_dtype == GPTQ_W_BF16)
    return launch_dt<__nv_bfloat16>(tq, tw, tg, qzeros, scales, r, c, bits, n_groups, st, stall, wait_ns);
  return launch_dt<__half>(tq, tw, tg, qzeros, scales, r, c, bits, n_groups, st, stall, wait_ns);
}

gptq_status_t launch_dequant(const int32_t* qweight, const int32_t* qzeros, const float* scales,
                             const int32_t* g_idx, int64_t d_row, int64_t d_col, int bits, int n_groups,
                             int out_dtype, void* W, cudaStream_t st) {
  return launch_dequant_impl(qweight, qzeros, scales, g_idx, d_row, d_col, bits, n_groups, out_dtype, W,
                             st, 0, kWaitLimitNs);
}

}  // namespace gptq

// Test hook (not part of the public header): the dequantization kernel
// launched with its producer stalled -- it issues no copy, so every bounded
// wait of the compute warps runs out after wait_ns and the kernel returns
// with GPTQ_ERR_TIMEOUT recorded in the library's fault word.  Nothing is in
// flight when the waits give up; used to test the timeout path.
extern "C" GPTQ_API int gptq_internal_dequant_stalled(const int32_t* qweight, const int32_t* qzeros,
                                                      const float* scales, const int32_t* g_idx,
                                                      int64_t d_row, int64_t d_col, int32_t bits,
                                                      int32_t group_size, void* W_out,
                                                      unsigned long long wait_ns,
                                                      gptq_stream_t stream) {
  if (!qweight || !qzeros || !scales || !g_idx || !W_out || d_row < 32 || d_row % 32 || d_col < 32 ||
      d_col % 32 || (bits != 2 && bits != 3 && bits != 4 && bits != 8) || wait_ns == 0)
    return GPTQ_ERR_INVALID_ARG;
  const int n_groups = group_size == -1 ? 1 : static_cast<int>(d_col / group_size);
  return gptq::launch_dequant_impl(qweight, qzeros, scales, g_idx, d_row, d_col, bits, n_groups,
                                   GPTQ_W_FP16, W_out, reinterpret_cast<cudaStream_t>(stream), 1,
                                   wait_ns);
}
