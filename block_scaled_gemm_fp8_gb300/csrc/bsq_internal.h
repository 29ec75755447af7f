// bsq_internal.h -- launch descriptions shared between the host entry points (bsq_api.cu)
// and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace bsq {

enum GemmOp : int { kDgrad = 0, kWgrad = 1, kBoth = 2 };   // kBoth: one launch, dgrad tiles then wgrad tiles

// Fixed tile shape of the fused kernel (see bsq_gemm.cu):
//   M side (tensor-memory lanes): 128 columns of the packed operand's contiguous axis
//   N side: up to 256 tokens (dgrad) or grad_out columns (wgrad)
//   K step: 64 rows of the packed operand per pipeline stage
constexpr int kTileM = 128;
constexpr int kTileN = 256;
constexpr int kTileK = 64;
constexpr int kMaxExperts = 1024;
constexpr int kMaxDevices = 64;   // device ordinals the per-device host state covers

// The kernels of a format: an FP8 weight with one scale per tensor runs the FP8 kernels,
// whose scale block is then the whole tensor (fp8_scale_shift).
inline int kernel_fmt(int fmt) { return fmt == 4 /* BSQ_FP8_E4M3_TENSOR */ ? 1 /* BSQ_FP8_E4M3_B128 */ : fmt; }
// log2 of the FP8 scale block's side: 7 for 128 x 128 blocks, 31 (every row and column
// index maps to block 0) for one scale per tensor.
inline int fp8_scale_shift(int fmt) { return fmt == 4 ? 31 : 7; }

struct GemmArgs {
  int op;            // kDgrad / kWgrad
  int fmt;           // bsq_format of the packed (dequantized) operand
  const void* p_data;
  const void* p_scale;
  const float* p_tensor_scale;
  int64_t p_batch;   // dgrad: E (weights per expert); wgrad: 1
  int64_t p_rows;    // rows of one packed matrix (dgrad: N; wgrad: S)
  int64_t kc;        // packed operand columns (K)
  const void* g;     // grad_out bf16 [S][N]
  int64_t S;
  int64_t N;
  const int32_t* offsets;  // device int32 [E] cumulative ends; nullptr = one group of S rows
  int64_t E;
  void* out;         // dgrad: bf16 [S][K]; wgrad: bf16 [E][N][K]
  int32_t* err;      // device error word
  int num_sms;
  cudaStream_t stream;
  int tail_rows;     // grouped dgrad: ragged last tiles of 1..tail_rows rows are left out
                     // (the small-M kernel's share, same rule); 0 = none
};

// Returns a cudaError_t-style code (0 = launched) and fills `msg` on failure.
int launch_gemm(const GemmArgs& a, const char** msg);
// One launch for a dgrad and a wgrad over the same grad_out (one packed format, one K):
// the dgrad's tiles, then the wgrad's.
int launch_gemm_backward(const GemmArgs& dgrad, const GemmArgs& wgrad, const char** msg);

struct DequantArgs {
  int fmt;
  const void* data;
  const void* scale;
  const float* tensor_scale;
  int64_t batch, rows, cols;
  void* out;
  int num_sms;
  cudaStream_t stream;
};

int launch_dequant(const DequantArgs& a, const char** msg);
// BSQ_FP8_E5M2_TENSOR codes with one float32 step per batch entry -> BF16 (bsq_quant.cu).
int launch_dequant_e5m2(const DequantArgs& a, const char** msg);

struct QuantArgs {
  const void* g;      // bf16 [n]
  int64_t n;
  int margin;         // 0..30
  void* codes;        // u8 [n] E5M2
  void* deq;          // bf16 [n] or nullptr
  float* step;        // f32 [1]
  float* amax;        // f32 [1]; also the reduction word
  int num_sms;
  cudaStream_t stream;
};
// Per-tensor E5M2 quantization with the current amax (bsq_quant.cu).
int launch_quantize_e5m2(const QuantArgs& a, const char** msg);

struct SmallMArgs {
  int fmt;
  const void* g;          // bf16 [M][N] (grouped: [S][N], M = S)
  const void* w_data;     // packed [N][K] (grouped: [E][N][K])
  const void* w_scale;
  const float* w_tensor_scale;   // NVFP4: f32[E]
  int64_t M, N, K;        // linear: M <= 16
  void* out;              // bf16 [M][K]
  void* ws;               // FP32 workspace of smallm_workspace_bytes(K) bytes, zero between calls
  int num_sms;
  cudaStream_t stream;
  int32_t* err;           // device error word
  const int32_t* offsets = nullptr;   // grouped (cluster kernel only): device cumulative ends [E]
  int64_t E = 1;
  int tail_rows = 0;      // grouped: rows of an expert taken (its ragged last GEMM tile, 1..tail_rows rows)
};

constexpr int kSmallM = 16;  // dgrad with at most this many rows takes the split-K kernel
size_t smallm_workspace_bytes(int64_t K);
int launch_smallm(const SmallMArgs& a, const char** msg);
// The same product with the row splits of a column slab reduced inside a thread-block
// cluster (distributed shared memory): no workspace (a.ws is not used).  With offsets it
// is the grouped dgrad of the rows that the pair-tile GEMM leaves out (GemmArgs::tail_rows).
int launch_smallm_cluster(const SmallMArgs& a, const char** msg);
// Grouped dgrad with at most this many grad_out rows in all goes wholly to the small-M
// kernel (BSQ_GROUPED_SMALL_ROWS overrides, 0..255; 0 never).
constexpr int kGroupedSmallRows = 64;
int grouped_small_rows();
// Above that, an expert's ragged last pair tile of at most this many rows goes to the
// small-M kernel and the rest to the GEMM (BSQ_GROUPED_TAIL_ROWS, 0..255; default 0: the
// GEMM takes every row).
int grouped_tail_rows();

struct ForwardArgs {
  int x_fmt, w_fmt;        // packed formats of X and W (one kernel format: kernel_fmt equal)
  const void* x_data;      // packed [M][K]
  const void* x_scale;
  const float* x_tensor_scale;
  const void* w_data;      // packed [N][K]
  const void* w_scale;
  const float* w_tensor_scale;
  int64_t M, N, K;
  void* y;                 // bf16 [M][N]
  int32_t* err;
  int num_sms;
  cudaStream_t stream;
};
// Y = deq(X) @ deq(W)^T (bsq_forward.cu).
int launch_forward(const ForwardArgs& a, const char** msg);

// Host-side argument checks of bsq_linear_dgrad (bsq_api.cu); BSQ_OK when well formed.
int check_linear_dgrad_args(const void* grad_out, int64_t M, int64_t N, int32_t w_fmt, const void* w_data,
                            const void* w_scale, const float* w_tensor_scale, int64_t K, const void* grad_x);
// The current device's error word and SM count (no allocation); BSQ_OK on success.
int device_error_word(int32_t** err, int* sms);
// Record a message for bsq_last_error() and return `status`.
int set_error(int status, const char* message);

// Wait limit of every pipeline wait inside the kernels (nanoseconds of %globaltimer),
// read from the environment at every call: BSQ_WAIT_LIMIT_US, else BSQ_WAIT_LIMIT_MS,
// else 2 s.
uint64_t wait_limit_ns();
// Limit of the waits an aborting kernel makes for its own copies and MMAs still in flight
// (they complete in microseconds; the limit only guards against a copy that never does).
constexpr uint64_t kDrainLimitNs = 2000000000ull;
// Time an aborting CTA pair leaves for asynchronous stores between its CTAs to land.
constexpr uint64_t kAbortSettleNs = 50000ull;

}  // namespace bsq
