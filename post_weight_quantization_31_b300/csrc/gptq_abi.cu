// The C ABI (include/gptq.h): argument checks, workspace sizes, status
// read-back, and the sticky device fault word.
#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace gptq {

uint64_t g_launches = 0;

__device__ int g_fault_word = 0;

namespace {
std::mutex g_fault_mu;
int* g_fault_addr[64] = {nullptr};
}  // namespace

int* fault_word_ptr() {
  // One address per device (the symbol lives in this library's module),
  // looked up on first use with that device current.
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_fault_mu);
  if (!g_fault_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fault_word) == cudaSuccess) g_fault_addr[dev] = static_cast<int*>(p);
  }
  return g_fault_addr[dev];
}

gptq_status_t launch_hessian_syrk(const void* X, int64_t d, int64_t n_tok, int64_t ldx, bool tok_major,
                                  float* S, cudaStream_t st);
gptq_status_t launch_diag_sumsq(const void* X, int64_t d, int64_t n_tok, int64_t ldx, bool tok_major,
                                double* diag, cudaStream_t st);
size_t prep_workspace_bytes(int64_t d);
gptq_status_t launch_prepare(const float* S, const double* diag, int64_t d, int64_t n_seen, float damp,
                             bool desc_act, float* U, int32_t* perm, void* ws, cudaStream_t st);
size_t quant_workspace_bytes(int64_t d_row, int64_t d_col);
gptq_status_t launch_quantize(const void* W, int w_dtype, int64_t d_row, int64_t d_col, const float* U,
                              const int32_t* perm, const gptq_config_t& cfg, uint8_t* codes,
                              float* scales, uint8_t* zeros, int32_t* g_idx, void* ws,
                              cudaStream_t st);
gptq_status_t launch_pack(const uint8_t* codes, const uint8_t* zeros, int64_t d_row, int64_t d_col,
                          int bits, int n_groups, int32_t* qweight, int32_t* qzeros, cudaStream_t st);
gptq_status_t launch_unpack(const int32_t* qweight, const int32_t* qzeros, int64_t d_row, int64_t d_col,
                            int bits, int n_groups, uint8_t* codes, uint8_t* zeros, cudaStream_t st);
size_t awq_workspace_bytes(int64_t d_row, int64_t d_col, int n_grid);
gptq_status_t launch_awq(const void* W, int w_dtype, int64_t d_row, int64_t d_col, const float* S,
                         const double* diag, const gptq_config_t& cfg, float frac, const float* grid_host,
                         int n_grid, uint8_t* codes, float* scales, uint8_t* zeros, float* t_out,
                         double* errors_out, void* ws, cudaStream_t st);
gptq_status_t launch_dequant(const int32_t* qweight, const int32_t* qzeros, const float* scales,
                             const int32_t* g_idx, int64_t d_row, int64_t d_col, int bits, int n_groups,
                             int out_dtype, void* W, cudaStream_t st);
gptq_status_t launch_dequant_matmul(const void* X, int x_dtype, int64_t M, int64_t ldx, const int32_t* qweight,
                                    const int32_t* qzeros, const float* scales, const int32_t* g_idx,
                                    int64_t d_row, int64_t d_col, int bits, int n_groups, float* Y,
                                    cudaStream_t st);

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool bits_ok(int bits) { return bits == 2 || bits == 3 || bits == 4 || bits == 8; }

bool config_ok(const gptq_config_t* c, int64_t d_col) {
  if (!c) return false;
  if (!bits_ok(c->bits)) return false;
  // The lazy-batch width only orders the same sums differently; the kernels
  // run their own 128 / 512-column blocking, whatever this value is.
  if (c->blocksize < 32 || c->blocksize % 32 != 0) return false;
  if (!(c->damp_percent >= 0.f) || !std::isfinite(c->damp_percent)) return false;
  if (c->desc_act != 0 && c->desc_act != 1) return false;
  if (c->sym != 0 && c->sym != 1) return false;
  const int gs = c->group_size;
  if (gs == -1) return true;
  if (gs <= 0 || gs % 32 != 0) return false;
  if (128 % gs != 0) return false;   // a group lies inside one 128-column block of the kernels
  if (d_col % gs != 0) return false;
  return true;
}

bool device_ok() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  return major == 10 && minor == 3;
}

int n_groups_of(int group_size, int64_t d_col) {
  return group_size == -1 ? 1 : static_cast<int>(d_col / group_size);
}

gptq_status_t status_of_bits(int bits) {
  if (bits & kStatTimeout) return GPTQ_ERR_TIMEOUT;
  if (bits & kStatNonFinite) return GPTQ_ERR_NONFINITE;
  if (bits & kStatNotPD) return GPTQ_ERR_NOT_PD;
  return GPTQ_OK;
}

// Reads (and clears) the library's sticky fault word; synchronizes the stream.
gptq_status_t read_fault_word(cudaStream_t st) {
  int fault = 0;
  int* fw = fault_word_ptr();
  if (!fw) return GPTQ_ERR_CUDA;
  if (cudaMemcpyAsync(&fault, fw, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return GPTQ_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return GPTQ_ERR_CUDA;
  if (fault) {
    if (cudaMemsetAsync(fw, 0, sizeof(int), st) != cudaSuccess) return GPTQ_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return GPTQ_ERR_CUDA;
    return GPTQ_ERR_TIMEOUT;
  }
  return GPTQ_OK;
}

}  // namespace

// The status word a prepare or quantize call leaves at the start of its
// workspace (offset 0 in both workspace layouts); synchronizes the stream.
gptq_status_t read_workspace_status(const void* ws, cudaStream_t st) {
  int bits = 0;
  if (cudaMemcpyAsync(&bits, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return GPTQ_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return GPTQ_ERR_CUDA;
  return status_of_bits(bits);
}

namespace {

}  // namespace
}  // namespace gptq

using namespace gptq;


extern "C" {

gptq_status_t gptq_hessian_accumulate(const void* X, int64_t d_col, int64_t n_tok, int64_t ldx,
                                      int32_t x_token_major, float* S, double* diag, int64_t* n_seen,
                                      gptq_stream_t stream) {
  if (!X || !S) return GPTQ_ERR_INVALID_ARG;
  if (x_token_major != 0 && x_token_major != 1) return GPTQ_ERR_INVALID_ARG;
  const bool tok = x_token_major != 0;
  if (d_col < 32 || d_col % 32 != 0 || n_tok < 1 || ldx % 8 != 0 || ldx < (tok ? d_col : n_tok))
    return GPTQ_ERR_INVALID_ARG;
  if (d_col > 46336 || n_tok > (int64_t(1) << 28)) return GPTQ_ERR_INVALID_ARG;
  if (!aligned(X, 16) || !aligned(S, 16) || (diag && !aligned(diag, 8))) return GPTQ_ERR_INVALID_ARG;
  if (!device_ok()) return GPTQ_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  gptq_status_t s = launch_hessian_syrk(X, d_col, n_tok, ldx, tok, S, st);
  if (s != GPTQ_OK) return s;
  if (diag) {
    s = launch_diag_sumsq(X, d_col, n_tok, ldx, tok, diag, st);
    if (s != GPTQ_OK) return s;
  }
  if (n_seen) *n_seen += n_tok;
  return GPTQ_OK;
}

size_t gptq_prepare_workspace_size(int64_t d_col) {
  if (d_col <= 0) return 0;
  return prep_workspace_bytes(d_col);
}


gptq_status_t gptq_prepare_hinv(const float* S, const double* diag, int64_t d_col, int64_t n_seen,
                                const gptq_config_t* cfg, float* U, int32_t* perm, void* ws,
                                size_t ws_bytes, gptq_stream_t stream) {
  if (!S || !U || !perm) return GPTQ_ERR_INVALID_ARG;
  if (d_col < 32 || d_col % 32 != 0 || d_col > 46336 || n_seen < 1) return GPTQ_ERR_INVALID_ARG;
  if (!config_ok(cfg, d_col)) return GPTQ_ERR_INVALID_ARG;
  if (!aligned(S, 16) || !aligned(U, 16) || !aligned(perm, 4) || (diag && !aligned(diag, 8)))
    return GPTQ_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256) || ws_bytes < prep_workspace_bytes(d_col)) return GPTQ_ERR_WORKSPACE;
  if (!device_ok()) return GPTQ_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return launch_prepare(S, diag, d_col, n_seen, cfg->damp_percent, cfg->desc_act != 0, U, perm, ws,
                        st);
}

size_t gptq_quantize_workspace_size(int64_t d_row, int64_t d_col, const gptq_config_t* cfg) {
  (void)cfg;
  if (d_row <= 0 || d_col <= 0) return 0;
  return quant_workspace_bytes(d_row, d_col);
}

gptq_status_t gptq_quantize_layer(const void* W, int32_t w_dtype, int64_t d_row, int64_t d_col,
                                  const float* U, const int32_t* perm, const gptq_config_t* cfg,
                                  uint8_t* codes, float* scales, uint8_t* zeros, int32_t* g_idx,
                                  void* ws, size_t ws_bytes, gptq_stream_t stream) {
  if (!W || !U || !perm || !codes || !scales || !zeros || !g_idx) return GPTQ_ERR_INVALID_ARG;
  if (w_dtype != GPTQ_W_FP32 && w_dtype != GPTQ_W_BF16 && w_dtype != GPTQ_W_FP16)
    return GPTQ_ERR_INVALID_ARG;
  if (d_row < 32 || d_row % 32 != 0 || d_col < 32 || d_col % 32 != 0) return GPTQ_ERR_INVALID_ARG;
  if (d_row * d_col > (int64_t(1) << 31) - 1 || d_col > 46336) return GPTQ_ERR_INVALID_ARG;
  if (!config_ok(cfg, d_col)) return GPTQ_ERR_INVALID_ARG;
  if (!aligned(W, 16) || !aligned(U, 16) || !aligned(scales, 4)) return GPTQ_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256) || ws_bytes < quant_workspace_bytes(d_row, d_col))
    return GPTQ_ERR_WORKSPACE;
  if (!device_ok()) return GPTQ_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return launch_quantize(W, w_dtype, d_row, d_col, U, perm, *cfg, codes, scales, zeros, g_idx, ws,
                         st);
}

size_t gptq_awq_workspace_size(int64_t d_row, int64_t d_col, int32_t n_grid) {
  if (d_row <= 0 || d_col <= 0 || n_grid <= 0) return 0;
  return awq_workspace_bytes(d_row, d_col, n_grid);
}

gptq_status_t gptq_awq_search(const void* W, int32_t w_dtype, int64_t d_row, int64_t d_col, const float* S,
                              const double* diag, const gptq_config_t* cfg, float salient_frac,
                              const float* grid, int32_t n_grid, uint8_t* codes, float* scales,
                              uint8_t* zeros, float* t, double* errors, void* ws, size_t ws_bytes,
                              gptq_stream_t stream) {
  if (!W || !S || !diag || !cfg || !grid || !codes || !scales || !zeros || !t) return GPTQ_ERR_INVALID_ARG;
  if (w_dtype != GPTQ_W_FP32 && w_dtype != GPTQ_W_BF16 && w_dtype != GPTQ_W_FP16) return GPTQ_ERR_INVALID_ARG;
  if (d_row < 32 || d_row % 32 != 0 || d_col < 32 || d_col % 32 != 0 || d_col > 46336) return GPTQ_ERR_INVALID_ARG;
  if (d_row * d_col > (int64_t(1) << 31) - 1) return GPTQ_ERR_INVALID_ARG;
  if (!bits_ok(cfg->bits) || (cfg->sym != 0 && cfg->sym != 1)) return GPTQ_ERR_INVALID_ARG;
  const int gs = cfg->group_size;
  if (gs != -1 && (gs <= 0 || gs % 32 != 0 || d_col % gs != 0)) return GPTQ_ERR_INVALID_ARG;
  if (!(salient_frac > 0.f) || salient_frac > 1.f) return GPTQ_ERR_INVALID_ARG;
  if (n_grid < 1 || n_grid > 256) return GPTQ_ERR_INVALID_ARG;
  for (int i = 0; i < n_grid; ++i)
    if (!(grid[i] > 0.f) || !std::isfinite(grid[i])) return GPTQ_ERR_INVALID_ARG;
  if (!aligned(W, 16) || !aligned(S, 16) || !aligned(diag, 8) || !aligned(scales, 4) || !aligned(t, 4) ||
      (errors && !aligned(errors, 8)))
    return GPTQ_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256) || ws_bytes < awq_workspace_bytes(d_row, d_col, n_grid)) return GPTQ_ERR_WORKSPACE;
  if (!device_ok()) return GPTQ_ERR_UNSUPPORTED;
  return launch_awq(W, w_dtype, d_row, d_col, S, diag, *cfg, salient_frac, grid, n_grid, codes, scales, zeros,
                    t, errors, ws, reinterpret_cast<cudaStream_t>(stream));
}

gptq_status_t gptq_pack(const uint8_t* codes, const uint8_t* zeros, int64_t d_row, int64_t d_col,
                        int32_t bits, int32_t group_size, int32_t* qweight, int32_t* qzeros,
                        gptq_stream_t stream) {
  if (!codes || !zeros || !qweight || !qzeros) return GPTQ_ERR_INVALID_ARG;
  if (!bits_ok(bits) || d_row < 32 || d_row % 32 != 0 || d_col < 32 || d_col % 32 != 0)
    return GPTQ_ERR_INVALID_ARG;
  if (group_size != -1 && (group_size <= 0 || d_col % group_size != 0)) return GPTQ_ERR_INVALID_ARG;
  if (d_row * d_col > (int64_t(1) << 31) - 1) return GPTQ_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(qweight, 4) || !aligned(qzeros, 4)) return GPTQ_ERR_INVALID_ARG;
  if (!device_ok()) return GPTQ_ERR_UNSUPPORTED;
  return launch_pack(codes, zeros, d_row, d_col, bits, n_groups_of(group_size, d_col), qweight, qzeros,
                     reinterpret_cast<cudaStream_t>(stream));
}

gptq_status_t gptq_unpack(const int32_t* qweight, const int32_t* qzeros, int64_t d_row, int64_t d_col,
                          int32_t bits, int32_t group_size, uint8_t* codes, uint8_t* zeros,
                          gptq_stream_t stream) {
  if (!codes || !zeros || !qweight || !qzeros) return GPTQ_ERR_INVALID_ARG;
  if (!bits_ok(bits) || d_row < 32 || d_row % 32 != 0 || d_col < 32 || d_col % 32 != 0)
    return GPTQ_ERR_INVALID_ARG;
  if (group_size != -1 && (group_size <= 0 || d_col % group_size != 0)) return GPTQ_ERR_INVALID_ARG;
  if (d_row * d_col > (int64_t(1) << 31) - 1) return GPTQ_ERR_INVALID_ARG;
  if (!aligned(qweight, 4) || !aligned(qzeros, 4)) return GPTQ_ERR_INVALID_ARG;
  if (!device_ok()) return GPTQ_ERR_UNSUPPORTED;
  return launch_unpack(qweight, qzeros, d_row, d_col, bits, n_groups_of(group_size, d_col), codes, zeros,
                       reinterpret_cast<cudaStream_t>(stream));
}

gptq_status_t gptq_dequantize(const int32_t* qweight, const int32_t* qzeros, const float* scales,
                              const int32_t* g_idx, int64_t d_row, int64_t d_col, int32_t bits,
                              int32_t group_size, int32_t out_dtype, void* W_out, gptq_stream_t stream) {
  if (!qweight || !qzeros || !scales || !g_idx || !W_out) return GPTQ_ERR_INVALID_ARG;
  if (!bits_ok(bits) || d_row < 32 || d_row % 32 != 0 || d_col < 32 || d_col % 32 != 0)
    return GPTQ_ERR_INVALID_ARG;
  if (group_size != -1 && (group_size <= 0 || d_col % group_size != 0)) return GPTQ_ERR_INVALID_ARG;
  if (out_dtype != GPTQ_W_FP32 && out_dtype != GPTQ_W_BF16 && out_dtype != GPTQ_W_FP16)
    return GPTQ_ERR_INVALID_ARG;
  if (d_row * d_col > (int64_t(1) << 31) - 1) return GPTQ_ERR_INVALID_ARG;
  if (!aligned(qweight, 16) || !aligned(qzeros, 4) || !aligned(scales, 4) || !aligned(g_idx, 16) ||
      !aligned(W_out, 16))
    return GPTQ_ERR_INVALID_ARG;
  if (!device_ok()) return GPTQ_ERR_UNSUPPORTED;
  return launch_dequant(qweight, qzeros, scales, g_idx, d_row, d_col, bits, n_groups_of(group_size, d_col),
                        out_dtype, W_out, reinterpret_cast<cudaStream_t>(stream));
}

gptq_status_t gptq_dequant_matmul(const void* X, int32_t x_dtype, int64_t M, int64_t ldx,
                                  const int32_t* qweight, const int32_t* qzeros, const float* scales,
                                  const int32_t* g_idx, int64_t d_row, int64_t d_col, int32_t bits,
                                  int32_t group_size, float* Y, gptq_stream_t stream) {
  if (!X || !qweight || !qzeros || !scales || !g_idx || !Y) return GPTQ_ERR_INVALID_ARG;
  if (x_dtype != GPTQ_W_FP16 && x_dtype != GPTQ_W_BF16) return GPTQ_ERR_INVALID_ARG;
  if (!bits_ok(bits) || d_row < 32 || d_row % 32 != 0 || d_col < 64 || d_col % 64 != 0)
    return GPTQ_ERR_INVALID_ARG;
  if (group_size != -1 && (group_size <= 0 || d_col % group_size != 0)) return GPTQ_ERR_INVALID_ARG;
  if (M < 1 || ldx < d_col || ldx % 8 != 0) return GPTQ_ERR_INVALID_ARG;
  if (M * d_row > (int64_t(1) << 31) - 1 || d_row * d_col > (int64_t(1) << 31) - 1 ||
      M * ldx > (int64_t(1) << 40))
    return GPTQ_ERR_INVALID_ARG;
  if (!aligned(X, 16) || !aligned(qweight, 16) || !aligned(g_idx, 16) || !aligned(qzeros, 4) ||
      !aligned(scales, 16) || !aligned(Y, 4))
    return GPTQ_ERR_INVALID_ARG;
  if (!device_ok()) return GPTQ_ERR_UNSUPPORTED;
  return launch_dequant_matmul(X, x_dtype, M, ldx, qweight, qzeros, scales, g_idx, d_row, d_col, bits,
                               n_groups_of(group_size, d_col), Y, reinterpret_cast<cudaStream_t>(stream));
}

const char* gptq_status_string(gptq_status_t s) {
  switch (s) {
    case GPTQ_OK: return "ok";
    case GPTQ_ERR_INVALID_ARG: return "invalid argument";
    case GPTQ_ERR_NOT_PD: return "damped Hessian is not positive definite (raise damp_percent)";
    case GPTQ_ERR_NONFINITE: return "non-finite value in the input";
    case GPTQ_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case GPTQ_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
    case GPTQ_ERR_CUDA: return "CUDA runtime error";
    case GPTQ_ERR_UNSUPPORTED: return "device is not sm_103 (B300)";
  }
  return "unknown status";
}

gptq_status_t gptq_device_fault(gptq_stream_t stream) {
  return read_fault_word(reinterpret_cast<cudaStream_t>(stream));
}

gptq_status_t gptq_workspace_status(const void* ws, gptq_stream_t stream) {
  if (!ws || !aligned(ws, 256)) return GPTQ_ERR_INVALID_ARG;
  return read_workspace_status(ws, reinterpret_cast<cudaStream_t>(stream));
}

uint64_t gptq_launch_count(void) { return __atomic_load_n(&g_launches, __ATOMIC_RELAXED); }

}  // extern "C"
