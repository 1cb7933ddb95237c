// gptq_prepare_hinv_noalloc: the prepare step with its scratch space in a
// fixed array that the library itself holds in device memory, for callers
// that cannot allocate device memory (see include/gptq.h).
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it until the process exits.  Host code cannot pass the
// array's name to a kernel (on the host that name is only a stand-in, not a
// device address), so the device address is looked up once per device with
// cudaGetSymbolAddress and cached.
#include <mutex>

#include "common.cuh"

namespace gptq {

size_t prep_workspace_bytes(int64_t d);
gptq_status_t read_workspace_status(const void* ws, cudaStream_t st);

namespace {

constexpr int64_t kMaxDCol = GPTQ_NOALLOC_MAX_D_COL;
constexpr size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
// Room for the prepare workspace at d_col = kMaxDCol: the status word, the
// per-block sums of the diagonal, the 64-bit sort keys, the low parts of the
// work matrix's diagonal, the d x d work matrix, the 128 x 128 inverse of a
// diagonal block, and two pairs of d x 128 panel operands.  Each call checks
// it against prep_workspace_bytes().
constexpr size_t kScratchBytes = 256 + round256(8 * (kMaxDCol / 256 + 1)) + round256(8 * kMaxDCol) +
                                 round256(4 * kMaxDCol) +
                                 round256(4 * kMaxDCol * kMaxDCol) + round256(4 * 128 * 128) +
                                 4 * round256(4 * kMaxDCol * 128);

static __device__ __align__(256) unsigned char g_prep_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {nullptr};

// Device address of g_prep_scratch on the current device (looked up on the
// first call per device).  Returns nullptr if the lookup fails.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_prep_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace
}  // namespace gptq

extern "C" GPTQ_API gptq_status_t gptq_prepare_hinv_noalloc(const float* S, const double* diag,
                                                            int64_t d_col, int64_t n_seen,
                                                            const gptq_config_t* cfg, float* U,
                                                            int32_t* perm, gptq_stream_t stream) {
  if (d_col > gptq::kMaxDCol) return GPTQ_ERR_WORKSPACE;
  if (d_col > 0 && gptq::prep_workspace_bytes(d_col) > gptq::kScratchBytes) return GPTQ_ERR_WORKSPACE;
  void* ws = gptq::scratch_address();
  if (!ws) return GPTQ_ERR_CUDA;
  const gptq_status_t s =
      gptq_prepare_hinv(S, diag, d_col, n_seen, cfg, U, perm, ws, gptq::kScratchBytes, stream);
  if (s != GPTQ_OK) return s;
  // The status word of the call sits in the library's array, where the
  // caller cannot read it: wait for the call and report it here.
  return gptq::read_workspace_status(ws, reinterpret_cast<cudaStream_t>(stream));
}
