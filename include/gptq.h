/*
 * gptq.h -- C ABI of the GPTQ per-layer weight-quantization solver for
 * NVIDIA B300 (sm_103a).
 *
 * The solver quantizes one linear layer W [d_row, d_col] (out_features x
 * in_features) to bits-wide integer codes with one scale and zero point per
 * group of input columns, using the layer's calibration activations
 * X [d_col, n_tok].  It is split into four calls that run back to back on
 * one CUDA stream:
 *
 *   gptq_hessian_accumulate   S += X X^T                          (step a1)
 *   gptq_prepare_hinv         H = 2/n S + damping, column order,
 *                             U with H^-1 = U^T U                  (step a2)
 *   gptq_quantize_layer       column loop with error feedback and
 *                             128-column lazy batch updates        (a3, a4)
 *   gptq_pack                 codes -> int32 words                 (step a5)
 *
 * Sources for what each step computes (web pages on GPTQ):
 *   [G] GPTQ practical guide, m.lqnn.cn/news/117696: §2.1 "从OBQ说起"
 *       (OBQ update, Hessian from calibration activations), §2.2 "固定顺序、
 *       Lazy Batch、Cholesky", §3.3 "量化超参怎么设置" (bits, group_size,
 *       desc_act, damp_percent), §3.4 (saving the packed model), §5.2
 *       (desc_act column re-order at load time).
 *   [S] "AWQ与GPTQ谁更强？ms-swift量化模块深度评测", GPTQ section
 *       (GptqConfig with sym=True).
 *   [E] "大模型压缩量化技术：GPTQ 与 AWQ 原理详解 + Python 实战教程", §二
 *       (min-max round-to-nearest grid), FAQ Q6 (group_size = -1).
 *
 * Conventions for every call:
 *   - All array arguments are DEVICE pointers (memory the caller allocated
 *     on the current CUDA device), unless the comment says "host".  The
 *     library never allocates device memory; scratch space is queried with
 *     the *_workspace_size functions and passed in by the caller.
 *   - Matrices are row-major and densely packed unless a leading dimension
 *     is given.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and every call returns once it is enqueued, without waiting
 *     for the GPU: the calls are stream-ordered and asynchronous, so the
 *     solves of several layers can run concurrently on several streams.
 *     Only gptq_workspace_status, gptq_device_fault and
 *     gptq_prepare_hinv_noalloc wait for their stream.
 *   - Argument errors are detected on the host before anything is enqueued
 *     and return GPTQ_ERR_INVALID_ARG (or GPTQ_ERR_WORKSPACE) with no side
 *     effect.  A CUDA error at launch returns GPTQ_ERR_CUDA.
 *   - Errors found on the device (a non-positive pivot, non-finite input, a
 *     wait that ran out) by gptq_prepare_hinv or gptq_quantize_layer are
 *     recorded in a status word at the start of that call's workspace; read
 *     it with gptq_workspace_status(ws, stream) after the call.  Each call
 *     clears its own word when it starts, so the word describes the last
 *     call that used the workspace, and a fault in one call never shows up
 *     in another's.
 *   - Every wait inside a kernel is bounded in time (about 2 s).  A wait that
 *     runs out makes its kernel return early and records GPTQ_ERR_TIMEOUT:
 *     in the call's workspace status word for gptq_prepare_hinv and
 *     gptq_quantize_layer; for the calls without a workspace (hessian,
 *     dequantize, dequant-matmul) in the library's per-device fault word,
 *     which gptq_device_fault reads and clears.  That word is shared by all
 *     streams of the device: a timeout there can stop, and is reported to,
 *     whichever of those calls runs or checks next.
 *   - Only one device is used per call: the current device of the calling
 *     host thread.
 */
#ifndef GPTQ_B300_H
#define GPTQ_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GPTQ_API __attribute__((visibility("default")))
#else
#define GPTQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, spelled without the CUDA headers. */
typedef struct CUstream_st* gptq_stream_t;

/*
 * Quantizer knobs, mirroring BaseQuantizeConfig / GptqConfig on the pages
 * ([G] §3.3, [S]).
 *   bits          2, 3, 4 or 8.
 *   group_size    columns sharing one scale and zero point, counted in
 *                 processing order: 32, 64 or 128 (a divisor of d_col);
 *                 or -1 for one group per row ([E] FAQ Q6).
 *   damp_percent  >= 0; lambda = damp_percent * mean(diag H) is added to
 *                 diag(H) ([G] §3.3, "防止矩阵奇异").
 *   blocksize     lazy-batch width ([G] §2.2): any positive multiple of 32.
 *                 Batching only changes the order in which the same
 *                 compensation terms are summed (the result is the same in
 *                 exact arithmetic), so the kernels keep their own two-level
 *                 blocking -- 128-column blocks inside 512-column super-blocks
 *                 -- and results agree with any blocksize up to fp32
 *                 rounding.
 *   desc_act      0: natural column order; 1: descending diag(H), stable.
 *   sym           0: asymmetric grid over [min(0,min w), max(0,max w)];
 *                 1: symmetric grid, scale 2*max|w|/maxq, zero (maxq+1)/2.
 */
typedef struct {
  int32_t bits;
  int32_t group_size;
  float damp_percent;
  int32_t blocksize;
  int32_t desc_act;
  int32_t sym;
} gptq_config_t;

typedef enum {
  GPTQ_OK = 0,
  GPTQ_ERR_INVALID_ARG = 1, /* bad size, knob, alignment or null pointer */
  GPTQ_ERR_NOT_PD = 2,      /* damped H has a non-positive pivot: retry with a
                               larger damp_percent (the pages' remedy, [G]
                               §3.3 and the 0.1 damping advice) */
  GPTQ_ERR_NONFINITE = 3,   /* NaN or Inf in S or W */
  GPTQ_ERR_WORKSPACE = 4,   /* workspace pointer null or too small */
  GPTQ_ERR_TIMEOUT = 5,     /* a bounded wait inside a kernel ran out */
  GPTQ_ERR_CUDA = 6,        /* CUDA runtime error (launch, copy, device) */
  GPTQ_ERR_UNSUPPORTED = 7  /* device is not sm_103 */
} gptq_status_t;

/* Storage type of W given to gptq_quantize_layer. */
enum { GPTQ_W_FP32 = 0, GPTQ_W_BF16 = 1, GPTQ_W_FP16 = 2 };

/*
 * a1  S += X X^T   ([G] §2.1: the Hessian is computed from the layer's
 *                   calibration activations; H = 2/n S is formed in a2.)
 *   X       fp16, read only, 16-byte aligned, ldx % 8 == 0:
 *           x_token_major = 0: [d_col, n_tok] with row stride ldx elements
 *             (tokens contiguous), ldx >= n_tok;
 *           x_token_major = 1: [n_tok, d_col] with row stride ldx elements
 *             (channels contiguous, the layout of a [tokens, features]
 *             activation tensor), ldx >= d_col.
 *           Both layouts feed the tensor cores directly (K-major or
 *           MN-major operand tiles); the result is the same up to the order
 *           of fp32 additions.
 *   S       fp32 [d_col, d_col], row-major, 16-byte aligned, updated in place
 *           with the full symmetric product (both triangles).  Zero it
 *           before the first call; call once per chunk of tokens.
 *   diag    fp64 [d_col] or NULL: if given, diag[i] += sum_t X[i,t]^2 computed
 *           to about 1e-14 relative (double-float sums on the fp32 ALUs).
 *           gptq_prepare_hinv takes the act-order (desc_act) column order
 *           from it, so that near-equal diagonals are ordered as exact
 *           arithmetic orders them; an fp32 diagonal would reorder them.
 *           Zero it with S.  Costs one extra read of X.
 *   n_seen  HOST pointer, may be NULL: *n_seen += n_tok on success.
 *   d_col % 32 == 0, d_col >= 32, n_tok >= 1.
 *   S runs on the 5th-generation tensor cores (fp16 x fp16 -> fp32).  The
 *   fp32 sums are added with atomics, so the order of additions, and hence
 *   the last bits of S, can differ from run to run.  Asynchronous.
 */
GPTQ_API gptq_status_t gptq_hessian_accumulate(const void* X, int64_t d_col, int64_t n_tok,
                                               int64_t ldx, int32_t x_token_major, float* S,
                                               double* diag, int64_t* n_seen, gptq_stream_t stream);

/* Bytes of workspace gptq_prepare_hinv needs for d_col. */
GPTQ_API size_t gptq_prepare_workspace_size(int64_t d_col);

/*
 * a2  From S and the token count n_seen: H = (2/n_seen) S;
 *     H += damp_percent * mean(diag H) * I; if desc_act, perm = stable
 *     argsort of -diag(H) ([G] §2.2 fixed order, §3.3 desc_act), else the
 *     identity; then U, upper triangular with positive diagonal, such that
 *     H[perm][:,perm]^-1 = U^T U ([G] §2.2 Cholesky reformulation).
 *   S       fp32 [d_col, d_col] from gptq_hessian_accumulate; only the lower
 *           triangle (i >= j) is read.  Read only.
 *   diag    fp64 [d_col] from gptq_hessian_accumulate, or NULL.  When given
 *           it supplies the diagonal of H, the damping mean and the desc_act
 *           order; otherwise the fp32 diagonal of S is used for all three.
 *           (The fp32 diagonal of S is biased low by a few 1e-6 relative; the
 *           fp64 one makes U about 10x closer to exact on wide layers.)
 *   U       fp32 [d_col, d_col] output, rows and columns in processing
 *           order; entries below the diagonal are written as 0.
 *   perm    int32 [d_col] output: perm[i] = original column processed i-th.
 *   ws      workspace of at least gptq_prepare_workspace_size(d_col) bytes,
 *           256-byte aligned.
 *   Asynchronous.  Device-side errors land in the status word of ws
 *   (gptq_workspace_status): GPTQ_ERR_NOT_PD for a non-positive pivot (U is
 *   then undefined; retry with a larger damp_percent), GPTQ_ERR_NONFINITE
 *   for NaN/Inf in S, GPTQ_ERR_TIMEOUT for a wait that ran out.
 */
GPTQ_API gptq_status_t gptq_prepare_hinv(const float* S, const double* diag, int64_t d_col, int64_t n_seen,
                                const gptq_config_t* cfg, float* U, int32_t* perm,
                                void* ws, size_t ws_bytes, gptq_stream_t stream);

/*
 * gptq_prepare_hinv without a caller workspace.  The pages have no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory when they need the factor -- code that runs inside another
 * framework's memory pool and may not allocate outside it, or a
 * latency-critical path where cudaMalloc / cudaFree would synchronize the
 * device.  It computes exactly what gptq_prepare_hinv computes, with the
 * same arguments except ws / ws_bytes, and allocates nothing: the scratch
 * space is a fixed array of about 5.3 MB that the library keeps in device
 * memory on every GPU it is loaded on, until the process exits.
 *   d_col   at most GPTQ_NOALLOC_MAX_D_COL (1024); larger values return
 *           GPTQ_ERR_WORKSPACE with no side effect.  Other argument errors
 *           and status codes are those of gptq_prepare_hinv.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current).  Every call, from any
 *   thread or stream,
 *   shares the one array and leaves its contents behind: calls whose GPU
 *   work overlaps (two streams, two host threads) race and corrupt each
 *   other's results, so serialize them.  Synchronizes `stream`.
 */
#define GPTQ_NOALLOC_MAX_D_COL 1024
GPTQ_API gptq_status_t gptq_prepare_hinv_noalloc(const float* S, const double* diag, int64_t d_col,
                                                 int64_t n_seen, const gptq_config_t* cfg, float* U,
                                                 int32_t* perm, gptq_stream_t stream);

/* Bytes of workspace gptq_quantize_layer needs. */
GPTQ_API size_t gptq_quantize_workspace_size(int64_t d_row, int64_t d_col, const gptq_config_t* cfg);

/*
 * a3 + a4  Quantize W column by column in processing order with OBQ error
 *     feedback ([G] §2.1; update w_F -= (w_j - dq_j)/U_jj * U[j, F]) and
 *     128-column lazy batches ([G] §2.2; after each block,
 *     W[:, i2:] -= Err U[i1:i2, i2:]).  At the first column of each group the
 *     group's scale and zero point are set from the group's current,
 *     error-updated values: span = max - min over the group's range
 *     (asymmetric; the range always includes 0) or 2 max|w| (symmetric),
 *     s = span / maxq, and
 *     code = clamp(rint(w / s) + z, 0, maxq), maxq = 2^bits - 1,
 *     round half to even, with w / s taken as maxq * (w / span) and w / span
 *     rounded as IEEE fp32 division rounds it (so a weight exactly halfway
 *     between two levels, like -max|w| on the symmetric grid, is decided as
 *     a tie).
 *   W       [d_row, d_col] of type w_dtype (GPTQ_W_FP32/BF16/FP16), 16-byte
 *           aligned.  Read only (the fp32 working copy lives in ws).
 *   U, perm outputs of gptq_prepare_hinv for the same cfg.
 *   codes   uint8 [d_row, d_col] output, ORIGINAL column order.
 *   scales  fp32  [G, d_row] output, G = d_col/group_size (1 if -1); group
 *           g covers processing positions [g*gs, (g+1)*gs).
 *   zeros   uint8 [G, d_row] output.
 *   g_idx   int32 [d_col] output: group of each original column.
 *   ws      workspace of gptq_quantize_workspace_size bytes, 256-byte aligned.
 *   d_row % 32 == 0, d_col % 32 == 0.  Asynchronous: GPTQ_ERR_NONFINITE for
 *   NaN/Inf in W and GPTQ_ERR_TIMEOUT land in the status word of ws
 *   (gptq_workspace_status).
 */
GPTQ_API gptq_status_t gptq_quantize_layer(const void* W, int32_t w_dtype, int64_t d_row,
                                  int64_t d_col, const float* U, const int32_t* perm,
                                  const gptq_config_t* cfg, uint8_t* codes, float* scales,
                                  uint8_t* zeros, int32_t* g_idx, void* ws, size_t ws_bytes,
                                  gptq_stream_t stream);

/*
 * a5  Pack codes and zero points into int32 words.  The pages only say the
 *     result is saved in "GPTQ format" with safetensors ([G] §3.4); this
 *     layout is the library's own:
 *   qweight int32 [d_col*bits/32, d_row]: column r holds row r's codes as an
 *           LSB-first bit stream along the input dimension (word k of row r
 *           holds columns [k*32/bits, (k+1)*32/bits) for bits 2, 4, 8; for
 *           bits 3, words 3m..3m+2 hold columns [32m, 32m+32) as one stream).
 *   qzeros  int32 [G, d_row*bits/32]: row g is zeros[g, :] as an LSB-first
 *           stream along d_row.
 *   codes / zeros values are masked to `bits` bits.  d_row % 32 == 0,
 *   d_col % 32 == 0.  Asynchronous.
 */
GPTQ_API gptq_status_t gptq_pack(const uint8_t* codes, const uint8_t* zeros, int64_t d_row,
                        int64_t d_col, int32_t bits, int32_t group_size, int32_t* qweight,
                        int32_t* qzeros, gptq_stream_t stream);

/* Inverse of gptq_pack (same layouts).  Asynchronous. */
GPTQ_API gptq_status_t gptq_unpack(const int32_t* qweight, const int32_t* qzeros, int64_t d_row,
                          int64_t d_col, int32_t bits, int32_t group_size, uint8_t* codes,
                          uint8_t* zeros, gptq_stream_t stream);

/* Bytes of workspace gptq_awq_search needs for d_row x d_col and n_grid
 * candidate factors. */
GPTQ_API size_t gptq_awq_workspace_size(int64_t d_row, int64_t d_col, int32_t n_grid);

/*
 * AWQ scale search, the activation-aware alternative to the GPTQ solve
 * ("大模型压缩量化技术：GPTQ 与 AWQ 原理详解", §四 AWQ 原理; "GPTQ/AWQ量化导出",
 * AWQ steps).  The channels whose activations are largest -- the
 * ceil(salient_frac * d_col) largest RMS sqrt(sum_t x^2 / n), ties to the
 * lower index -- have their weights multiplied by one factor s before
 * round-to-nearest quantization (the GPTQ grid of cfg, group-wise in
 * natural column order); the effective weights are the dequantized values
 * divided by s, and at inference those activations are divided by s.  s is
 * the candidate in `grid` with the smallest layer output error
 * tr(D S D^T), D = W - effective weights (the earliest on ties).
 *   W        [d_row, d_col] of w_dtype, 16-byte aligned.  Read only.
 *   S, diag  from gptq_hessian_accumulate over the layer's calibration
 *            tokens (diag, the fp64 sums of squares, is required).
 *   cfg      bits, group_size (32, 64, 128 dividing d_col, or -1) and sym;
 *            the other fields are not used.
 *   salient_frac  in (0, 1]; 0.05 on the pages.
 *   grid     HOST array of n_grid (1..256) positive candidate factors, e.g.
 *            1, 1.25, ..., 4 (1 keeps plain round-to-nearest among them).
 *   codes    uint8 [d_row, d_col] output: codes of W diag(t), natural order
 *            (g_idx[c] = c / group_size for gptq_pack's consumers).
 *   scales   fp32 [G, d_row], zeros uint8 [G, d_row] outputs (of W diag(t)).
 *   t        fp32 [d_col] output: s for the salient channels, 1 elsewhere.
 *   errors   fp64 [n_grid] device output (may be NULL): each candidate's
 *            error tr(D S D^T), with S as given (so in units of X X^T).
 *   ws       gptq_awq_workspace_size bytes, 256-byte aligned.
 *   Asynchronous; a wait that runs out lands in the status word of ws
 *   (gptq_workspace_status).  The error products run on the tensor cores
 *   (3xTF32, fp32-accurate) and are summed in fp64.
 */
GPTQ_API gptq_status_t gptq_awq_search(const void* W, int32_t w_dtype, int64_t d_row, int64_t d_col,
                                       const float* S, const double* diag, const gptq_config_t* cfg,
                                       float salient_frac, const float* grid, int32_t n_grid,
                                       uint8_t* codes, float* scales, uint8_t* zeros, float* t,
                                       double* errors, void* ws, size_t ws_bytes, gptq_stream_t stream);

/*
 * The packed layer back to dense weights, in the ORIGINAL column order:
 *   W_out[r][c] = scales[g][r] * (code[r][c] - zero[g][r]),  g = g_idx[c],
 * formed in fp32 and rounded to nearest in out_dtype (GPTQ_W_FP32 / _BF16 /
 * _FP16).  With desc_act the columns of a group are scattered and g_idx
 * re-orders them, as the guide's §5.2 says happens when such a model is
 * loaded ([G] §5.2); this is the consumer that checks the packed format
 * end to end.
 *   qweight, qzeros  layouts of gptq_pack; qweight 16-byte aligned.
 *   scales           fp32 [G, d_row].
 *   g_idx            int32 [d_col], 16-byte aligned, values in [0, G)
 *                    (others are clamped into range, so the result is then
 *                    undefined but no memory outside the arrays is read).
 *   W_out            [d_row, d_col] of out_dtype, 16-byte aligned.
 *   d_row % 32 == 0, d_col % 32 == 0, group_size as in gptq_pack.
 *   All pointers are device memory owned by the caller.  Asynchronous;
 *   GPTQ_ERR_INVALID_ARG for bad sizes, types or alignment.  The kernel's
 *   internal waits are bounded: if one runs out, the library's fault flag
 *   is set and the next gptq_device_fault() (or synchronizing call)
 *   returns GPTQ_ERR_TIMEOUT.
 */
GPTQ_API gptq_status_t gptq_dequantize(const int32_t* qweight, const int32_t* qzeros, const float* scales,
                                       const int32_t* g_idx, int64_t d_row, int64_t d_col, int32_t bits,
                                       int32_t group_size, int32_t out_dtype, void* W_out,
                                       gptq_stream_t stream);

/*
 * Y = X · Wᵀ with W the packed layer, dequantized on the fly: the matmul a
 * GPTQ layer runs at inference, unpacking the codes to 16-bit weights and
 * multiplying ([G] §4.3), with the desc_act column order resolved through
 * g_idx ([G] §5.2).  W[n][k] = scales[g][n]·(code[n][k] − zero[g][n]),
 * g = g_idx[k], formed in fp32 and rounded to X's type (the same values
 * gptq_dequantize writes for that type); the products are summed in fp32 on
 * the tensor cores.  The order of the sums is the kernel's: results agree
 * with an exact product of the same operands to within
 * (d_col + 148)·2⁻²³·Σ_k |X[m][k]·W[n][k]|.
 *   X        [M, ldx] of x_dtype (GPTQ_W_FP16 or GPTQ_W_BF16), the first
 *            d_col entries of each row used; 16-byte aligned, ldx % 8 == 0.
 *   qweight, qzeros, scales, g_idx   as for gptq_dequantize (qweight,
 *            scales and g_idx 16-byte aligned).  d_row = output features
 *            (N), d_col = input features (K).
 *   Y        fp32 [M, d_row], overwritten.
 *   d_row % 32 == 0, d_col % 64 == 0, M >= 1, group_size as in gptq_pack.
 *   All pointers are device memory owned by the caller.  Asynchronous;
 *   GPTQ_ERR_INVALID_ARG for bad sizes, types or alignment.  Internal waits
 *   are bounded as for gptq_dequantize.
 */
GPTQ_API gptq_status_t gptq_dequant_matmul(const void* X, int32_t x_dtype, int64_t M, int64_t ldx,
                                           const int32_t* qweight, const int32_t* qzeros,
                                           const float* scales, const int32_t* g_idx, int64_t d_row,
                                           int64_t d_col, int32_t bits, int32_t group_size, float* Y,
                                           gptq_stream_t stream);

/* Static English text for a status code. */
GPTQ_API const char* gptq_status_string(gptq_status_t status);

/* Synchronizes `stream`; returns GPTQ_ERR_TIMEOUT (and clears the flag) if a
 * bounded wait ran out since the last check in a kernel of a call that has
 * no workspace (hessian, dequantize, dequant-matmul), else GPTQ_OK (or
 * GPTQ_ERR_CUDA). */
GPTQ_API gptq_status_t gptq_device_fault(gptq_stream_t stream);

/*
 * Waits for `stream` (cudaStreamSynchronize), then returns the status that
 * the last gptq_prepare_hinv or gptq_quantize_layer call using the
 * workspace `ws` (device pointer, the same one passed to that call) left in
 * it: GPTQ_OK, GPTQ_ERR_NOT_PD, GPTQ_ERR_NONFINITE or GPTQ_ERR_TIMEOUT.
 * `stream` must be the call's stream (or one ordered after it).  The word is
 * left as it is; the next call on the workspace clears it when it starts.
 */
GPTQ_API gptq_status_t gptq_workspace_status(const void* ws, gptq_stream_t stream);

/* Number of kernels this library has launched in this process (all
 * devices); for instrumentation. */
GPTQ_API uint64_t gptq_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* GPTQ_B300_H */
