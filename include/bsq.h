/*
 * bsq.h -- C ABI of libbsq: the backward pass of block-scaled low-precision linear
 * layers and of their grouped (mixture-of-experts) form, on one GB300 GPU (sm_103a).
 *
 * What is computed (the "dequantize, then BF16 matmul" backward):
 *   MSLK PR #393 "Add Autograd Backward Support for FP4 GEMM Custom Ops",
 *   section "Implementation Method": saved packed FP4 operands are dequantized to
 *   BF16 and the standard gradients are taken,
 *       grad_X = grad_out @ W_bf16        grad_W = grad_out^T @ X_bf16
 *   transformers PR #50031 "Train adapters on top of FP8 weights":
 *   `_dequantize_fp8_weight` (E4M3 weights, float32 scale_inv per 128x128 block,
 *   scale cast to the gradient dtype), `FP8LinearFunction.backward` (dgrad only,
 *   the FP8 weight is frozen) and `FP8GroupedMatmulFunction.backward` (grouped dgrad
 *   over int32 expert offsets).
 *
 * Dequantization rule (bit-exact): out = RNE_bf16( bf16(code value) * RNE_bf16(scale) ).
 *   FP8 E4M3      scale = scale_inv[b][r/128][c/128]                         (float32)
 *   FP8 E4M3, one scale per tensor:  scale = scale_inv[b]                      (float32)
 *   MXFP4         scale = 2^(e8m0[b][r][c/32] - 127), byte 255 = NaN
 *   NVFP4         scale = RNE_fp32( e4m3[b][r][c/16] * tensor_scale[b] )
 * FP4 packing: byte j of a row holds element 2j in bits 0-3 and 2j+1 in bits 4-7.
 * The GEMMs accumulate in FP32 (tensor cores) and round the result once to BF16.
 *
 * Conventions shared by every entry point
 *   - All pointers except `code` in bsq_get_device_error are DEVICE pointers into
 *     the current CUDA device's memory; the caller allocates and owns every buffer.
 *     Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default).
 *   - Tensors are dense and row-major: [batch][rows][cols], cols contiguous.
 *   - Packed operand of format `fmt`:
 *       BSQ_BF16           data bf16[batch][rows][cols]; scale, tensor_scale unused
 *       BSQ_FP8_E4M3_B128  data u8  [batch][rows][cols];
 *                          scale f32[batch][ceil(rows/128)][ceil(cols/128)]
 *       BSQ_FP8_E4M3_TENSOR data u8 [batch][rows][cols]; scale f32[batch] (one scale_inv per
 *                          tensor -- per expert for a grouped weight -- broadcast over it:
 *                          transformers PR #50031 `_dequantize_fp8_weight`, block_size None)
 *       BSQ_FP8_E5M2_TENSOR data u8 [batch][rows][cols] E5M2 codes; scale f32[batch] (one
 *                          quantization step per tensor, bsq_quantize_e5m2); dequantized by
 *                          the same rule with the step as the scale
 *       BSQ_MXFP4          data u8  [batch][rows][cols/2]; scale u8 [batch][rows][cols/32]
 *       BSQ_NVFP4          data u8  [batch][rows][cols/2]; scale u8 (E4M3) [batch][rows][cols/16];
 *                          tensor_scale f32[batch]
 *   - Alignment: data/scale base pointers 16-byte aligned; the row pitch of every
 *     TMA-read tensor a multiple of 16 bytes, i.e. N % 8 == 0 for grad_out, and
 *     K % 16 (both FP8 formats), K % 32 (MXFP4, NVFP4), K % 8 (BF16) for the packed operand;
 *     a per-tensor FP8 scale array needs only 4-byte alignment.
 *     M, S and the expert sizes are arbitrary.
 *   - Errors: every call validates its arguments on the host first and returns a
 *     status without launching anything when they are wrong.  Nothing is thrown.
 *     BSQ_ERR_UNSUPPORTED marks a well-formed request the library does not serve
 *     (an alignment above, too many experts); BSQ_ERR_CUDA a failed launch.
 *     Device-side conditions (decreasing offsets, a pipeline wait that ran out of
 *     time) are recorded in a per-device error word read by bsq_get_device_error.
 *   - Allocation: the caller owns every tensor.  The library allocates no device memory:
 *     its own device state is one error word per device and the split-K scratch of
 *     bsq_linear_dgrad_smallm_noalloc, both file-scope device arrays of the library.
 *   - Environment (read by the host side at every call; none changes a result beyond FP32
 *     summation order):
 *       BSQ_WAIT_LIMIT_US,    bound of every pipeline wait inside a kernel, in microseconds
 *       BSQ_WAIT_LIMIT_MS     or milliseconds (the first one set wins; default 2000 ms); on
 *                             expiry the kernel lets its own copies and MMAs in flight finish,
 *                             writes nothing more, returns and records BSQ_DEVERR_TIMEOUT; the
 *                             outputs of that call are then undefined.
 *       BSQ_GEMM_SHORT_TILES  wgrad of a packed format: 1 = the short-tile GEMM kernel (more
 *                             epilogue warps), 0 = the default kernel; unset = the short-tile
 *                             kernel when the groups average fewer than 1024 rows (S < 1024*E).
 *       BSQ_GROUPED_SMALL_ROWS grouped dgrad of a packed W with S at most this many rows
 *                             (0..255, default 64) runs wholly in the split-K small-M kernel
 *                             (decode-sized batches); above it the pair-tile GEMM runs.
 *       BSQ_GROUPED_TAIL_ROWS above that bound, an expert's ragged last GEMM tile of at most
 *                             this many rows (0..255, default 0 = none) goes to the small-M
 *                             kernel instead; the two kernels then run one after the other.
 *       BSQ_TEST_DROP_ANNOUNCE test hook for failure detection: 1 = in the GEMM and forward
 *                             kernels, the even CTA of each pair never announces a unit's operands, so the
 *                             MMA thread's wait runs out of time (BSQ_WAIT_LIMIT_*), the kernel
 *                             stops in order and records BSQ_DEVERR_TIMEOUT.  Never set it
 *                             outside such a test: every GEMM and forward call then fails.
 *       BSQ_TEST_DROP_CHUNK   the same for the small-M kernel (bsq_linear_dgrad with M <= 16,
 *                             decode-sized bsq_grouped_dgrad): every CTA's first chunk is
 *                             never requested, so the wait for it runs out.
 */
#ifndef BSQ_H
#define BSQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BSQ_OK = 0,
  BSQ_ERR_INVALID_ARG = 1,
  BSQ_ERR_UNSUPPORTED = 2,
  BSQ_ERR_CUDA = 3,
  BSQ_ERR_TIMEOUT = 4
} bsq_status;

typedef enum {
  BSQ_BF16 = 0,
  BSQ_FP8_E4M3_B128 = 1,
  BSQ_MXFP4 = 2,
  BSQ_NVFP4 = 3,
  BSQ_FP8_E4M3_TENSOR = 4,
  BSQ_FP8_E5M2_TENSOR = 5   /* the quantized gradient: bsq_dequant only, not a GEMM operand */
} bsq_format;

/* Device error word values (bsq_get_device_error). */
#define BSQ_DEVERR_NONE 0
#define BSQ_DEVERR_TIMEOUT 1      /* a pipeline wait exceeded its time limit; the kernel returned early */
#define BSQ_DEVERR_BAD_OFFSETS 2  /* offsets decreasing, negative or beyond S; no output was written */

/*
 * bsq_dequant -- decode a packed operand to BF16 (the standalone dequantization the
 * transformers PR #50031 `_dequantize_fp8_weight` performs; MSLK PR #393's FP4
 * dequantization helpers).  out: bf16[batch][rows][cols].  fmt must not be BSQ_BF16.
 * Requirements: cols % 16 == 0 (both FP8 formats), cols % 32 == 0 (MXFP4), cols % 16 == 0 (NVFP4).
 */
bsq_status bsq_dequant(int32_t fmt, const void* data, const void* scale, const float* tensor_scale,
                       int64_t batch, int64_t rows, int64_t cols, void* out, void* stream);

/*
 * bsq_linear_dgrad -- grad_x[M][K] = grad_out[M][N] @ deq(W)[N][K]
 * (MSLK PR #393, Implementation Method; transformers PR #50031 FP8LinearFunction.backward).
 * grad_out: bf16[M][N]; W: packed [1][N][K] in w_fmt; grad_x: bf16[M][K] (fully written).
 * M <= 16 with a packed W takes a split-K kernel whose row splits add their partial sums
 * inside a thread-block cluster (distributed shared memory): no workspace, so such calls
 * may run concurrently on different streams.
 */
bsq_status bsq_linear_dgrad(const void* grad_out, int64_t M, int64_t N,
                            int32_t w_fmt, const void* w_data, const void* w_scale,
                            const float* w_tensor_scale, int64_t K, void* grad_x, void* stream);

/*
 * bsq_linear_wgrad -- grad_w[N][K] = grad_out[M][N]^T @ deq(X)[M][K]
 * (MSLK PR #393, Implementation Method).  X: packed [1][M][K] in x_fmt (BSQ_BF16 allowed).
 * grad_w: bf16[N][K] (fully written; M == 0 gives zeros).
 */
bsq_status bsq_linear_wgrad(const void* grad_out, int64_t M, int64_t N,
                            int32_t x_fmt, const void* x_data, const void* x_scale,
                            const float* x_tensor_scale, int64_t K, void* grad_w, void* stream);

/* Bits of `needs` in bsq_linear_backward: which gradients the caller wants. */
#define BSQ_NEEDS_GRAD_X 1u   /* grad_x = grad_out @ deq(W) */
#define BSQ_NEEDS_GRAD_W 2u   /* grad_w = grad_out^T @ deq(X) */

/*
 * bsq_linear_backward -- both gradients of a linear layer from one grad_out, with output
 * masks: AstrAI `astrai/extension/fp8.py`, `_LinearFp8.backward` (the gradient is shared by
 * dX and dW; `ctx.needs_input_grad` decides which of the two products run), applied to the
 * dequantize-then-BF16-matmul backward of MSLK PR #393, Implementation Method:
 *     grad_x[M][K] = grad_out[M][N] @ deq(W)[N][K]        (if needs & BSQ_NEEDS_GRAD_X)
 *     grad_w[N][K] = grad_out[M][N]^T @ deq(X)[M][K]      (if needs & BSQ_NEEDS_GRAD_W)
 * W: packed [1][N][K] in w_fmt; X: packed [1][M][K] in x_fmt (BSQ_BF16 allowed for either).
 * Arguments of a product that is not wanted are not read and may be null.  With both
 * products, the same packed format for W and X and M > 16, one persistent launch computes
 * the dgrad tiles and then the wgrad tiles, so grad_out streams through the L2 once for
 * both; otherwise the call behaves as bsq_linear_dgrad followed by bsq_linear_wgrad on the
 * stream.  Every output element equals the corresponding single-product entry point's
 * (the same tiles in the same accumulation order).  needs == 0 returns BSQ_OK and does
 * nothing; unknown bits return BSQ_ERR_INVALID_ARG.
 */
bsq_status bsq_linear_backward(const void* grad_out, int64_t M, int64_t N,
                               int32_t w_fmt, const void* w_data, const void* w_scale,
                               const float* w_tensor_scale,
                               int32_t x_fmt, const void* x_data, const void* x_scale,
                               const float* x_tensor_scale,
                               int64_t K, uint32_t needs, void* grad_x, void* grad_w, void* stream);

/*
 * bsq_linear_forward -- y[M][N] = deq(X)[M][K] @ deq(W)[N][K]^T, the forward product of the
 * layer the entry points above differentiate (MSLK PR #393, Summary: the mslk::f4f4bf16 ops
 * multiply packed X and W; the backward the PR adds is that of this product).  Both
 * operands are dequantized with the rule above, multiplied on the tensor cores with FP32
 * accumulation and rounded once to BF16.
 * X: packed [1][M][K] in x_fmt, W: packed [1][N][K] in w_fmt; W packed (not BSQ_BF16).  X is
 * either BSQ_BF16 (a BF16 activation, as in the FP8 linear layer of transformers PR #50031
 * whose weight alone is quantized: y = X @ deq(W)^T, K % 8 == 0) or packed of the same kind
 * as W: both FP4 of one format, or both FP8 (128x128 blocks or per tensor, mixed).
 * y: bf16[M][N], fully written; N % 8 == 0.  K == 0 gives zeros.
 */
bsq_status bsq_linear_forward(int32_t x_fmt, const void* x_data, const void* x_scale,
                              const float* x_tensor_scale, int64_t M,
                              int32_t w_fmt, const void* w_data, const void* w_scale,
                              const float* w_tensor_scale, int64_t N, int64_t K, void* y, void* stream);

/*
 * bsq_grouped_dgrad -- per expert e, grad_x[r0:r1] = grad_out[r0:r1] @ deq(W[e])
 * (transformers PR #50031 FP8GroupedMatmulFunction.backward).
 * offsets: device int32[E], cumulative END offsets without a leading zero
 * (expert e owns rows [e ? offsets[e-1] : 0, offsets[e])), non-decreasing, offsets[E-1] <= S.
 * W: packed [E][N][K]; w_tensor_scale (NVFP4) is per expert, f32[E].
 * grad_x: bf16[S][K]; rows >= offsets[E-1] of grad_x are not written, and the values of
 * grad_out there (possibly uninitialised) never reach a result.
 * 1 <= E <= 1024.
 * Kernels: with S <= 64 rows in all (BSQ_GROUPED_SMALL_ROWS) the split-K small-M kernel,
 * which reads every routed expert's packed weight once per 16 rows; else the pair-tile GEMM.
 */
bsq_status bsq_grouped_dgrad(const void* grad_out, int64_t S, int64_t N,
                             int32_t w_fmt, const void* w_data, const void* w_scale,
                             const float* w_tensor_scale, int64_t E, int64_t K,
                             const int32_t* offsets, void* grad_x, void* stream);

/*
 * bsq_grouped_wgrad -- per expert e, grad_w[e] = grad_out[r0:r1]^T @ deq(X)[r0:r1]
 * (MSLK PR #393, Implementation Method, applied per group).  X: packed [1][S][K].
 * grad_w: bf16[E][N][K], every expert written; an expert with no rows gets exact zeros.
 * Rows >= offsets[E-1] of grad_out and X are never read.  1 <= E <= 1024.
 */
bsq_status bsq_grouped_wgrad(const void* grad_out, int64_t S, int64_t N,
                             int32_t x_fmt, const void* x_data, const void* x_scale,
                             const float* x_tensor_scale, int64_t K, const int32_t* offsets,
                             int64_t E, void* grad_w, void* stream);

/*
 * bsq_linear_dgrad_smallm_noalloc -- the same product as bsq_linear_dgrad, for callers that
 * cannot allocate device memory (code running under stream capture, hosts whose allocator
 * owns all device memory, or processes that forbid allocation after start-up).  The pages
 * have no counterpart: it is an allocation-free variant of this library's split-K small-M
 * dgrad kernel that adds its row splits through global memory.  Its FP32 split-K scratch
 * is a file-scope device array of the library; every device that loads the library holds
 * that array (about 1 MiB) until the process exits.
 * Limits: 1 <= M <= 16, w_fmt FP8 (128x128 blocks) / MXFP4 / NVFP4, K <= 16384; anything else returns
 * BSQ_ERR_UNSUPPORTED (or the usual argument errors) without launching.
 * Allocation: calls no cudaMalloc / cudaFree or any allocating routine.  The first call on
 * a device looks up the array's device address (cudaGetSymbolAddress) with that device
 * current, and the address is kept for the life of the process; make that first call
 * before any stream capture.  A cudaDeviceReset invalidates the kept address: this entry
 * point is not to be called on a device after it was reset.
 * Sharing: every call uses the same array and clears the part it needs on `stream` before
 * its kernel; calls whose work overlaps on the GPU (different streams) race on the array
 * and must be ordered by the caller.
 */
bsq_status bsq_linear_dgrad_smallm_noalloc(const void* grad_out, int64_t M, int64_t N,
                                           int32_t w_fmt, const void* w_data, const void* w_scale,
                                           const float* w_tensor_scale, int64_t K, void* grad_x,
                                           void* stream);

/*
 * bsq_quantize_e5m2 -- per-tensor E5M2 quantization of a BF16 gradient with the current
 * amax (AstrAI fp8.py, `_LinearFp8.backward` in the "hybrid" format and `_dynamic_scale`):
 *   amax = max |g| (float32, at least 1e-12; NaN when g holds a NaN),
 *   step = (amax / 57344) / 2^margin   (float32 divisions),
 *   codes[i] = E5M2 of g[i] / step     (float32 division, nearest even, saturating to +-57344).
 * g: bf16[n], 16-byte aligned.  codes: u8[n], 8-byte aligned.  deq (optional, may be NULL):
 * bf16[n], 16-byte aligned, receives bf16(bf16(code) * bf16(step)) -- what bsq_dequant of
 * the codes gives.  step, amax: one f32 each (device); amax also serves as the kernels'
 * reduction word, so it must not alias step or the inputs.  0 <= margin <= 30.
 */
bsq_status bsq_quantize_e5m2(const void* g, int64_t n, int32_t margin, void* codes, void* deq, float* step,
                             float* amax, void* stream);

/*
 * bsq_linear_backward_e5m2 -- the backward with a quantized gradient: grad_out is quantized
 * once to E5M2 (bsq_quantize_e5m2 into g_codes, g_deq, g_step, g_amax) and both products
 * of bsq_linear_backward run on the dequantized copy g_deq (AstrAI fp8.py,
 * `_LinearFp8.backward`: one quantization shared by dX and dW, masks from
 * needs_input_grad, the gradient's amax returned for the caller's history).
 * g_codes u8[M][N] and g_deq bf16[M][N] are caller-owned scratch; the other arguments are
 * those of bsq_linear_backward.  Every operand check runs before anything is launched.
 */
bsq_status bsq_linear_backward_e5m2(const void* grad_out, int64_t M, int64_t N, int32_t w_fmt, const void* w_data,
                                    const void* w_scale, const float* w_tensor_scale, int32_t x_fmt,
                                    const void* x_data, const void* x_scale, const float* x_tensor_scale, int64_t K,
                                    uint32_t needs, int32_t margin, void* g_codes, void* g_deq, float* g_step,
                                    float* g_amax, void* grad_x, void* grad_w, void* stream);

/* Human-readable name of a status code (static string). */
const char* bsq_status_string(int32_t status);

/* Message describing the last failing call on this host thread ("" if none). */
const char* bsq_last_error(void);

/*
 * bsq_get_device_error -- synchronize `stream`, then read and clear the current
 * device's error word into *code (host pointer).  Returns BSQ_ERR_TIMEOUT when the
 * word held BSQ_DEVERR_TIMEOUT, BSQ_ERR_INVALID_ARG for BSQ_DEVERR_BAD_OFFSETS, else BSQ_OK.
 */
bsq_status bsq_get_device_error(int32_t* code, void* stream);

/* Number of SMs the persistent kernels are sized for on the current device (0 on error). */
int32_t bsq_num_sms(void);

#ifdef __cplusplus
}
#endif

#endif /* BSQ_H */
