// Step a5: packing codes and zero points into int32 words, and the inverse.
//
// The pages only say the quantized model is saved in "GPTQ format" next to
// a quantize_config.json ([G] GPTQ practical guide, m.lqnn.cn/news/117696,
// §3.4); the word layout below is this library's own:
//   qweight [d_col*bits/32, d_row]: column r of qweight is row r's codes as
//           an LSB-first bit stream along the input dimension;
//   qzeros  [G, d_row*bits/32]: row g is zeros[g, :] as an LSB-first stream.
// For 2, 4 and 8 bits a word holds 32/bits whole codes; for 3 bits every 3
// words hold 32 codes.
#include <algorithm>

#include "common.cuh"

namespace gptq {
namespace {

constexpr int PK_ROWS = 32;
constexpr int PK_COLS = 256;

// Word `kw` (LSB-first) of the bit stream of codes c[0..), each `bits` wide.
__device__ __forceinline__ uint32_t stream_word(const uint8_t* c, int stride, int kw, int bits,
                                                uint32_t mask) {
  uint32_t word = 0;
  const int b0 = 32 * kw;
  for (int i = b0 / bits; i * bits < b0 + 32; ++i) {
    const int sh = i * bits - b0;
    const uint32_t v = c[i * stride] & mask;
    word |= sh >= 0 ? (v << sh) : (v >> (-sh));
  }
  return word;
}

__global__ void pack_qweight_kernel(const uint8_t* __restrict__ codes, int d_row, int d_col, int bits,
                                    int32_t* __restrict__ qweight) {
  // Rows padded by one word: the 32 lanes below each read a different row
  // at the same column, and a 260-byte row stride puts those reads in 32
  // different banks (an unpadded 256-byte stride would put all of them in one).
  __shared__ __align__(16) uint8_t tile[PK_ROWS][PK_COLS + 4];
  const int r0 = blockIdx.y * PK_ROWS;
  const int c0 = blockIdx.x * PK_COLS;
  const int ncols = min(PK_COLS, d_col - c0);
  for (int idx = threadIdx.x; idx < PK_ROWS * (PK_COLS / 4); idx += blockDim.x) {
    const int rr = idx / (PK_COLS / 4), cc = (idx % (PK_COLS / 4)) * 4;
    uint32_t v = 0;
    if (r0 + rr < d_row && cc < ncols)
      v = *reinterpret_cast<const uint32_t*>(codes + static_cast<size_t>(r0 + rr) * d_col + c0 + cc);
    *reinterpret_cast<uint32_t*>(&tile[rr][cc]) = v;
  }
  __syncthreads();
  const uint32_t mask = (1u << bits) - 1u;
  const int words = ncols * bits / 32;
  const int wbase = c0 * bits / 32;
  for (int idx = threadIdx.x; idx < words * PK_ROWS; idx += blockDim.x) {
    const int rr = idx % PK_ROWS, kw = idx / PK_ROWS;
    if (r0 + rr >= d_row) continue;
    qweight[static_cast<size_t>(wbase + kw) * d_row + r0 + rr] =
        static_cast<int32_t>(stream_word(&tile[rr][0], 1, kw, bits, mask));
  }
}

// 2, 4 and 8 bits: a word holds whole codes, so each thread packs the 32
// codes of one row's 32-column chunk (two 16-byte loads, a whole sector)
// into `bits` words straight from registers; the lanes of a warp take 32
// consecutive rows, so every word store is one coalesced 128-byte line.
// The threads after those pack the zero points, one qzeros word each (the
// same launch, so the small qzeros work adds no launch of its own).
template <int BITS>
__global__ void pack_qweight_whole_kernel(const uint8_t* __restrict__ codes, int d_row, int d_col,
                                          int32_t* __restrict__ qweight,
                                          const uint8_t* __restrict__ zeros, int n_groups,
                                          int32_t* __restrict__ qzeros) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nq = static_cast<int64_t>(d_row) * (d_col / 32);
  if (gid >= nq) {
    const int words = d_row * BITS / 32;
    const int64_t zid = gid - nq;
    if (zid >= static_cast<int64_t>(words) * n_groups) return;
    const int g = static_cast<int>(zid / words), kw = static_cast<int>(zid % words);
    qzeros[static_cast<size_t>(g) * words + kw] = static_cast<int32_t>(
        stream_word(zeros + static_cast<size_t>(g) * d_row, 1, kw, BITS, (1u << BITS) - 1u));
    return;
  }
  const int r = static_cast<int>(gid % d_row);
  const int chunk = static_cast<int>(gid / d_row);
  const uint4* src = reinterpret_cast<const uint4*>(codes + static_cast<size_t>(r) * d_col + chunk * 32);
  const uint4 a = src[0], b = src[1];
  const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};  // 4 codes per word, one per byte
  int32_t* dst = qweight + static_cast<size_t>(chunk) * BITS * d_row + r;
  if constexpr (BITS == 8) {
#pragma unroll
    for (int j = 0; j < 8; ++j) dst[static_cast<size_t>(j) * d_row] = static_cast<int32_t>(u[j]);
  } else if constexpr (BITS == 4) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t w = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // 4 bytes -> 4 nibbles in the low 16 bits
        uint32_t t = u[2 * j + h] & 0x0F0F0F0Fu;
        t = (t | (t >> 4)) & 0x00FF00FFu;
        t = (t | (t >> 8)) & 0x0000FFFFu;
        w |= t << (16 * h);
      }
      dst[static_cast<size_t>(j) * d_row] = static_cast<int32_t>(w);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t w = 0;
#pragma unroll
      for (int h = 0; h < 4; ++h) {  // 4 bytes -> 4 two-bit fields in the low 8 bits
        uint32_t t = u[4 * j + h] & 0x03030303u;
        t = (t | (t >> 6)) & 0x000F000Fu;
        t = (t | (t >> 12)) & 0x000000FFu;
        w |= t << (8 * h);
      }
      dst[static_cast<size_t>(j) * d_row] = static_cast<int32_t>(w);
    }
  }
}

__global__ void pack_qzeros_kernel(const uint8_t* __restrict__ zeros, int d_row, int n_groups, int bits,
                                   int32_t* __restrict__ qzeros) {
  const int words = d_row * bits / 32;
  const int g = blockIdx.y;
  const uint32_t mask = (1u << bits) - 1u;
  for (int kw = blockIdx.x * blockDim.x + threadIdx.x; kw < words; kw += gridDim.x * blockDim.x)
    qzeros[static_cast<size_t>(g) * words + kw] =
        static_cast<int32_t>(stream_word(zeros + static_cast<size_t>(g) * d_row, 1, kw, bits, mask));
}

// Value of code i (bits wide) of the LSB-first stream held in words w[0..)
// with stride ws between consecutive words.
__device__ __forceinline__ uint8_t stream_get(const int32_t* w, size_t ws, int i, int bits) {
  const int b = i * bits;
  const int k = b >> 5, sh = b & 31;
  uint64_t v = static_cast<uint32_t>(w[k * ws]);
  if (sh + bits > 32) v |= static_cast<uint64_t>(static_cast<uint32_t>(w[(k + 1) * ws])) << 32;
  return static_cast<uint8_t>((v >> sh) & ((1u << bits) - 1u));
}

__global__ void unpack_qweight_kernel(const int32_t* __restrict__ qweight, int d_row, int d_col,
                                      int bits, uint8_t* __restrict__ codes) {
  for (int r = blockIdx.y; r < d_row; r += gridDim.y)
    for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < d_col; c += gridDim.x * blockDim.x)
      codes[static_cast<size_t>(r) * d_col + c] = stream_get(qweight + r, d_row, c, bits);
}

__global__ void unpack_qzeros_kernel(const int32_t* __restrict__ qzeros, int d_row, int bits,
                                     uint8_t* __restrict__ zeros) {
  const int g = blockIdx.y;
  const int words = d_row * bits / 32;
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < d_row; r += gridDim.x * blockDim.x)
    zeros[static_cast<size_t>(g) * d_row + r] =
        stream_get(qzeros + static_cast<size_t>(g) * words, 1, r, bits);
}

}  // namespace

gptq_status_t launch_pack(const uint8_t* codes, const uint8_t* zeros, int64_t d_row, int64_t d_col,
                          int bits, int n_groups, int32_t* qweight, int32_t* qzeros, cudaStream_t st) {
  if (bits != 3) {
    const int64_t threads = d_row * (d_col / 32) + d_row * bits / 32 * n_groups;   // d_col % 32 == 0
    const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
    const int dr = static_cast<int>(d_row), dc = static_cast<int>(d_col);
    if (bits == 8)
      pack_qweight_whole_kernel<8><<<blocks, 256, 0, st>>>(codes, dr, dc, qweight, zeros, n_groups, qzeros);
    else if (bits == 4)
      pack_qweight_whole_kernel<4><<<blocks, 256, 0, st>>>(codes, dr, dc, qweight, zeros, n_groups, qzeros);
    else
      pack_qweight_whole_kernel<2><<<blocks, 256, 0, st>>>(codes, dr, dc, qweight, zeros, n_groups, qzeros);
    GPTQ_LAUNCH_CHECK();
    return GPTQ_OK;
  }
  dim3 g1((d_col + PK_COLS - 1) / PK_COLS, (d_row + PK_ROWS - 1) / PK_ROWS);
  pack_qweight_kernel<<<g1, 256, 0, st>>>(codes, static_cast<int>(d_row), static_cast<int>(d_col), bits,
                                          qweight);
  GPTQ_LAUNCH_CHECK();
  const int words = static_cast<int>(d_row * bits / 32);
  dim3 g2((words + 255) / 256, n_groups);
  pack_qzeros_kernel<<<g2, 256, 0, st>>>(zeros, static_cast<int>(d_row), n_groups, bits, qzeros);
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

gptq_status_t launch_unpack(const int32_t* qweight, const int32_t* qzeros, int64_t d_row, int64_t d_col,
                            int bits, int n_groups, uint8_t* codes, uint8_t* zeros, cudaStream_t st) {
  dim3 g1(static_cast<unsigned>(std::min<int64_t>((d_col + 255) / 256, 64)), static_cast<unsigned>(std::min<int64_t>(d_row, 65535)));
  unpack_qweight_kernel<<<g1, 256, 0, st>>>(qweight, static_cast<int>(d_row), static_cast<int>(d_col),
                                            bits, codes);
  GPTQ_LAUNCH_CHECK();
  dim3 g2(static_cast<unsigned>((d_row + 255) / 256), n_groups);
  unpack_qzeros_kernel<<<g2, 256, 0, st>>>(qzeros, static_cast<int>(d_row), bits, zeros);
  GPTQ_LAUNCH_CHECK();
  return GPTQ_OK;
}

}  // namespace gptq
