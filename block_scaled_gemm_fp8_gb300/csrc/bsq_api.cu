// bsq_api.cu -- the C entry points declared in include/bsq.h: host-side argument
// validation, status codes, the per-device error word, and dispatch to the kernels.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "bsq_internal.h"
#include "../../include/bsq.h"

namespace {

thread_local char g_msg[512] = "";

// Per-device error word written by the kernels (BSQ_DEVERR_*); read and cleared by
// bsq_get_device_error.  One int per device, allocated with the module.
__device__ int32_t g_device_error;

using bsq::kMaxDevices;
int32_t* g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
std::mutex g_mu;

bsq_status fail(bsq_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
bsq_status fail(bsq_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}

// Device-specific set-up, done once per device with that device current.
bsq_status device_state(int32_t** err, int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(BSQ_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(BSQ_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) return fail(BSQ_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(BSQ_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
      return fail(BSQ_ERR_UNSUPPORTED, "libbsq is built for sm_103a; device %d is sm_%d%d", dev, major, minor);
    g_err_ptr[dev] = static_cast<int32_t*>(p);
    g_num_sms[dev] = n;
  }
  *err = g_err_ptr[dev];
  *sms = g_num_sms[dev];
  return BSQ_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared validation of a packed operand [batch][rows][cols].
bsq_status check_packed(const char* what, int32_t fmt, const void* data, const void* scale, const float* ts,
                        int64_t batch, int64_t rows, int64_t cols, bool allow_bf16) {
  if (fmt < BSQ_BF16 || fmt > BSQ_FP8_E5M2_TENSOR) return fail(BSQ_ERR_INVALID_ARG, "%s: unknown format %d", what, fmt);
  if (fmt == BSQ_BF16 && !allow_bf16) return fail(BSQ_ERR_UNSUPPORTED, "%s: BF16 is not a packed format here", what);
  if (batch < 0 || rows < 0 || cols < 0) return fail(BSQ_ERR_INVALID_ARG, "%s: negative size", what);
  const int64_t elems = batch * rows * cols;
  if (elems > 0 && !data) return fail(BSQ_ERR_INVALID_ARG, "%s: null data", what);
  if (elems > 0 && !aligned16(data)) return fail(BSQ_ERR_INVALID_ARG, "%s: data not 16-byte aligned", what);
  if (fmt != BSQ_BF16 && elems > 0 && !scale) return fail(BSQ_ERR_INVALID_ARG, "%s: null scale", what);
  if (fmt == BSQ_NVFP4 && elems > 0 && !ts) return fail(BSQ_ERR_INVALID_ARG, "%s: null tensor_scale", what);
  if (fmt == BSQ_FP8_E4M3_B128 && elems > 0 && !aligned16(scale))
    return fail(BSQ_ERR_INVALID_ARG, "%s: scale_inv not 16-byte aligned", what);
  if ((fmt == BSQ_FP8_E4M3_TENSOR || fmt == BSQ_FP8_E5M2_TENSOR) && elems > 0 && (reinterpret_cast<uintptr_t>(scale) & 3u))
    return fail(BSQ_ERR_INVALID_ARG, "%s: scale_inv not 4-byte aligned", what);
  switch (fmt) {
    case BSQ_BF16:
      if (cols % 8) return fail(BSQ_ERR_UNSUPPORTED, "%s: BF16 cols %% 8 != 0 (row pitch must be 16 bytes)", what);
      break;
    case BSQ_FP8_E4M3_B128:
    case BSQ_FP8_E4M3_TENSOR:
    case BSQ_FP8_E5M2_TENSOR:
      if (cols % 16) return fail(BSQ_ERR_UNSUPPORTED, "%s: FP8 cols %% 16 != 0 (row pitch must be 16 bytes)", what);
      break;
    case BSQ_MXFP4:
      if (cols % 32) return fail(BSQ_ERR_INVALID_ARG, "%s: MXFP4 cols %% 32 != 0", what);
      break;
    case BSQ_NVFP4:
      if (cols % 16) return fail(BSQ_ERR_INVALID_ARG, "%s: NVFP4 cols %% 16 != 0", what);
      break;
  }
  if (rows > INT32_MAX || cols > INT32_MAX || batch > INT32_MAX)
    return fail(BSQ_ERR_UNSUPPORTED, "%s: dimension above 2^31-1", what);
  return BSQ_OK;
}

// out_elems: elements of the output; an empty output may be null.
bsq_status check_gemm_common(const char* what, const void* g, int64_t S, int64_t N, int32_t fmt, int64_t K,
                             const void* out, int64_t out_elems) {
  if (S < 0 || N < 0 || K < 0) return fail(BSQ_ERR_INVALID_ARG, "%s: negative size", what);
  if (fmt == BSQ_FP8_E5M2_TENSOR)
    return fail(BSQ_ERR_UNSUPPORTED, "%s: E5M2 is the gradient's format (bsq_linear_backward_e5m2), not an operand's", what);
  if (S > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return fail(BSQ_ERR_UNSUPPORTED, "%s: size above 2^31-1", what);
  if (S * N > 0 && (!g || !aligned16(g))) return fail(BSQ_ERR_INVALID_ARG, "%s: grad_out null or not 16-byte aligned", what);
  if (N % 8) return fail(BSQ_ERR_UNSUPPORTED, "%s: N %% 8 != 0 (grad_out row pitch must be 16 bytes)", what);
  if (fmt == BSQ_NVFP4 && K % 32)
    return fail(BSQ_ERR_UNSUPPORTED, "%s: NVFP4 K %% 32 != 0 (packed row pitch must be 16 bytes)", what);
  if (out_elems > 0 && !out) return fail(BSQ_ERR_INVALID_ARG, "%s: null output", what);
  if (out_elems > 0 && !aligned16(out)) return fail(BSQ_ERR_INVALID_ARG, "%s: output not 16-byte aligned", what);
  return BSQ_OK;
}

bsq_status run_gemm(bsq::GemmArgs& a, const char* what) {
  int32_t* err = nullptr;
  int sms = 0;
  bsq_status st = device_state(&err, &sms);
  if (st != BSQ_OK) return st;
  a.err = err;
  a.num_sms = sms;
  const char* msg = "";
  if (bsq::launch_gemm(a, &msg) != 0) return fail(BSQ_ERR_CUDA, "%s: %s", what, msg);
  return BSQ_OK;
}

bsq_status zero_output(void* out, int64_t bytes, cudaStream_t s, const char* what) {
  if (bytes <= 0) return BSQ_OK;
  const cudaError_t e = cudaMemsetAsync(out, 0, static_cast<size_t>(bytes), s);
  if (e != cudaSuccess) return fail(BSQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return BSQ_OK;
}

}  // namespace

namespace bsq {
int check_linear_dgrad_args(const void* grad_out, int64_t M, int64_t N, int32_t w_fmt, const void* w_data,
                            const void* w_scale, const float* w_tensor_scale, int64_t K, const void* grad_x) {
  bsq_status st = check_gemm_common("bsq_linear_dgrad", grad_out, M, N, w_fmt, K, grad_x, M * K);
  if (st != BSQ_OK) return st;
  return check_packed("bsq_linear_dgrad", w_fmt, w_data, w_scale, w_tensor_scale, 1, N, K, true);
}
int device_error_word(int32_t** err, int* sms) { return device_state(err, sms); }
int set_error(int status, const char* message) {
  return fail(static_cast<bsq_status>(status), "%s", message);
}
uint64_t wait_limit_ns() {
  const char* us = std::getenv("BSQ_WAIT_LIMIT_US");
  const long u = us ? std::atol(us) : 0;
  if (u > 0) return static_cast<uint64_t>(u) * 1000ull;
  const char* ms = std::getenv("BSQ_WAIT_LIMIT_MS");
  const long m = ms ? std::atol(ms) : 0;
  return static_cast<uint64_t>(m > 0 ? m : 2000) * 1000000ull;
}
}  // namespace bsq

extern "C" {

const char* bsq_status_string(int32_t s) {
  switch (s) {
    case BSQ_OK: return "BSQ_OK";
    case BSQ_ERR_INVALID_ARG: return "BSQ_ERR_INVALID_ARG";
    case BSQ_ERR_UNSUPPORTED: return "BSQ_ERR_UNSUPPORTED";
    case BSQ_ERR_CUDA: return "BSQ_ERR_CUDA";
    case BSQ_ERR_TIMEOUT: return "BSQ_ERR_TIMEOUT";
    default: return "BSQ_ERR_UNKNOWN";
  }
}

const char* bsq_last_error(void) { return g_msg; }

int32_t bsq_num_sms(void) {
  int32_t* err = nullptr;
  int sms = 0;
  return device_state(&err, &sms) == BSQ_OK ? sms : 0;
}

bsq_status bsq_get_device_error(int32_t* code, void* stream) {
  if (!code) return fail(BSQ_ERR_INVALID_ARG, "bsq_get_device_error: null code");
  int32_t* err = nullptr;
  int sms = 0;
  bsq_status st = device_state(&err, &sms);
  if (st != BSQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(BSQ_ERR_CUDA, "bsq_get_device_error: %s", cudaGetErrorString(e));
  int32_t v = 0;
  e = cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(BSQ_ERR_CUDA, "bsq_get_device_error: %s", cudaGetErrorString(e));
  const int32_t zero = 0;
  e = cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fail(BSQ_ERR_CUDA, "bsq_get_device_error: %s", cudaGetErrorString(e));
  *code = v;
  if (v == BSQ_DEVERR_TIMEOUT) return fail(BSQ_ERR_TIMEOUT, "a kernel wait ran out of time");
  if (v == BSQ_DEVERR_BAD_OFFSETS) return fail(BSQ_ERR_INVALID_ARG, "offsets were not non-decreasing within [0, S]");
  return BSQ_OK;
}

bsq_status bsq_dequant(int32_t fmt, const void* data, const void* scale, const float* tensor_scale, int64_t batch,
                       int64_t rows, int64_t cols, void* out, void* stream) {
  bsq_status st = check_packed("bsq_dequant", fmt, data, scale, tensor_scale, batch, rows, cols, false);
  if (st != BSQ_OK) return st;
  if (batch * rows * cols == 0) return BSQ_OK;
  if (!out || !aligned16(out)) return fail(BSQ_ERR_INVALID_ARG, "bsq_dequant: output null or not 16-byte aligned");
  if (fmt == BSQ_MXFP4 && !aligned16(data)) return fail(BSQ_ERR_INVALID_ARG, "bsq_dequant: data alignment");
  int32_t* err = nullptr;
  int sms = 0;
  st = device_state(&err, &sms);
  if (st != BSQ_OK) return st;
  bsq::DequantArgs a{fmt, data, scale, tensor_scale, batch, rows, cols, out, sms, static_cast<cudaStream_t>(stream)};
  const char* msg = "";
  if ((fmt == BSQ_FP8_E5M2_TENSOR ? bsq::launch_dequant_e5m2(a, &msg) : bsq::launch_dequant(a, &msg)) != 0)
    return fail(BSQ_ERR_CUDA, "bsq_dequant: %s", msg);
  return BSQ_OK;
}

bsq_status bsq_linear_dgrad(const void* grad_out, int64_t M, int64_t N, int32_t w_fmt, const void* w_data,
                            const void* w_scale, const float* w_tensor_scale, int64_t K, void* grad_x,
                            void* stream) {
  const char* what = "bsq_linear_dgrad";
  bsq_status st = check_gemm_common(what, grad_out, M, N, w_fmt, K, grad_x, M * K);
  if (st != BSQ_OK) return st;
  st = check_packed(what, w_fmt, w_data, w_scale, w_tensor_scale, 1, N, K, true);
  if (st != BSQ_OK) return st;
  if (M == 0 || K == 0) return BSQ_OK;
  if (N == 0) return zero_output(grad_x, M * K * 2, static_cast<cudaStream_t>(stream), what);
  if (M <= bsq::kSmallM && w_fmt != BSQ_BF16) {
    // a few token rows: bound by reading W once; split-K kernel whose row splits add up
    // inside a thread-block cluster (no workspace)
    int32_t* err = nullptr;
    int sms = 0;
    st = device_state(&err, &sms);
    if (st != BSQ_OK) return st;
    bsq::SmallMArgs s{w_fmt, grad_out, w_data, w_scale, w_tensor_scale, M, N, K, grad_x, nullptr, sms,
                      static_cast<cudaStream_t>(stream), err};
    const char* msg = "";
    if (bsq::launch_smallm_cluster(s, &msg) != 0) return fail(BSQ_ERR_CUDA, "%s: %s", what, msg);
    return BSQ_OK;
  }
  bsq::GemmArgs a{};
  a.op = bsq::kDgrad; a.fmt = w_fmt; a.p_data = w_data; a.p_scale = w_scale; a.p_tensor_scale = w_tensor_scale;
  a.p_batch = 1; a.p_rows = N; a.kc = K; a.g = grad_out; a.S = M; a.N = N; a.offsets = nullptr; a.E = 1;
  a.out = grad_x; a.stream = static_cast<cudaStream_t>(stream);
  return run_gemm(a, what);
}

bsq_status bsq_linear_wgrad(const void* grad_out, int64_t M, int64_t N, int32_t x_fmt, const void* x_data,
                            const void* x_scale, const float* x_tensor_scale, int64_t K, void* grad_w,
                            void* stream) {
  const char* what = "bsq_linear_wgrad";
  bsq_status st = check_gemm_common(what, grad_out, M, N, x_fmt, K, grad_w, N * K);
  if (st != BSQ_OK) return st;
  st = check_packed(what, x_fmt, x_data, x_scale, x_tensor_scale, 1, M, K, true);
  if (st != BSQ_OK) return st;
  if (N == 0 || K == 0) return BSQ_OK;
  if (M == 0) return zero_output(grad_w, N * K * 2, static_cast<cudaStream_t>(stream), what);
  bsq::GemmArgs a{};
  a.op = bsq::kWgrad; a.fmt = x_fmt; a.p_data = x_data; a.p_scale = x_scale; a.p_tensor_scale = x_tensor_scale;
  a.p_batch = 1; a.p_rows = M; a.kc = K; a.g = grad_out; a.S = M; a.N = N; a.offsets = nullptr; a.E = 1;
  a.out = grad_w; a.stream = static_cast<cudaStream_t>(stream);
  return run_gemm(a, what);
}

bsq_status bsq_linear_backward(const void* grad_out, int64_t M, int64_t N, int32_t w_fmt, const void* w_data,
                               const void* w_scale, const float* w_tensor_scale, int32_t x_fmt, const void* x_data,
                               const void* x_scale, const float* x_tensor_scale, int64_t K, uint32_t needs,
                               void* grad_x, void* grad_w, void* stream) {
  const char* what = "bsq_linear_backward";
  if (needs & ~static_cast<uint32_t>(BSQ_NEEDS_GRAD_X | BSQ_NEEDS_GRAD_W))
    return fail(BSQ_ERR_INVALID_ARG, "%s: unknown bits in needs (0x%x)", what, needs);
  const bool want_x = (needs & BSQ_NEEDS_GRAD_X) != 0, want_w = (needs & BSQ_NEEDS_GRAD_W) != 0;
  if (!want_x && !want_w) return BSQ_OK;
  if (!want_w)
    return bsq_linear_dgrad(grad_out, M, N, w_fmt, w_data, w_scale, w_tensor_scale, K, grad_x, stream);
  if (!want_x)
    return bsq_linear_wgrad(grad_out, M, N, x_fmt, x_data, x_scale, x_tensor_scale, K, grad_w, stream);
  bsq_status st = check_gemm_common(what, grad_out, M, N, w_fmt, K, grad_x, M * K);
  if (st != BSQ_OK) return st;
  st = check_gemm_common(what, grad_out, M, N, x_fmt, K, grad_w, N * K);
  if (st != BSQ_OK) return st;
  st = check_packed(what, w_fmt, w_data, w_scale, w_tensor_scale, 1, N, K, true);
  if (st != BSQ_OK) return st;
  st = check_packed(what, x_fmt, x_data, x_scale, x_tensor_scale, 1, M, K, true);
  if (st != BSQ_OK) return st;
  // One launch for both products needs one packed format and enough token rows for the
  // tensor-core dgrad (fewer go to the small-M kernel); otherwise the two entry points run
  // one after the other on the stream.
  if (bsq::kernel_fmt(w_fmt) != bsq::kernel_fmt(x_fmt) || M <= bsq::kSmallM || N == 0 || K == 0 || M == 0) {
    st = bsq_linear_dgrad(grad_out, M, N, w_fmt, w_data, w_scale, w_tensor_scale, K, grad_x, stream);
    if (st != BSQ_OK) return st;
    return bsq_linear_wgrad(grad_out, M, N, x_fmt, x_data, x_scale, x_tensor_scale, K, grad_w, stream);
  }
  int32_t* err = nullptr;
  int sms = 0;
  st = device_state(&err, &sms);
  if (st != BSQ_OK) return st;
  bsq::GemmArgs d{};
  d.op = bsq::kDgrad; d.fmt = w_fmt; d.p_data = w_data; d.p_scale = w_scale; d.p_tensor_scale = w_tensor_scale;
  d.p_batch = 1; d.p_rows = N; d.kc = K; d.g = grad_out; d.S = M; d.N = N; d.offsets = nullptr; d.E = 1;
  d.out = grad_x; d.stream = static_cast<cudaStream_t>(stream); d.err = err; d.num_sms = sms;
  bsq::GemmArgs w = d;
  w.op = bsq::kWgrad; w.fmt = x_fmt; w.p_data = x_data; w.p_scale = x_scale; w.p_tensor_scale = x_tensor_scale;
  w.p_rows = M;
  w.out = grad_w;
  const char* msg = "";
  if (bsq::launch_gemm_backward(d, w, &msg) != 0) return fail(BSQ_ERR_CUDA, "%s: %s", what, msg);
  return BSQ_OK;
}

bsq_status bsq_linear_forward(int32_t x_fmt, const void* x_data, const void* x_scale, const float* x_tensor_scale,
                              int64_t M, int32_t w_fmt, const void* w_data, const void* w_scale,
                              const float* w_tensor_scale, int64_t N, int64_t K, void* y, void* stream) {
  const char* what = "bsq_linear_forward";
  if (M < 0 || N < 0 || K < 0) return fail(BSQ_ERR_INVALID_ARG, "%s: negative size", what);
  bsq_status st = check_packed(what, x_fmt, x_data, x_scale, x_tensor_scale, 1, M, K, true);
  if (st != BSQ_OK) return st;
  st = check_packed(what, w_fmt, w_data, w_scale, w_tensor_scale, 1, N, K, false);
  if (st != BSQ_OK) return st;
  if (x_fmt == BSQ_FP8_E5M2_TENSOR || w_fmt == BSQ_FP8_E5M2_TENSOR)
    return fail(BSQ_ERR_UNSUPPORTED, "%s: E5M2 is the gradient's format, not an operand's", what);
  if (x_fmt != BSQ_BF16 && bsq::kernel_fmt(x_fmt) != bsq::kernel_fmt(w_fmt))
    return fail(BSQ_ERR_UNSUPPORTED, "%s: X and W must share a packed format (FP8 blocks and per-tensor mix)", what);
  if (N % 8) return fail(BSQ_ERR_UNSUPPORTED, "%s: N %% 8 != 0 (Y row pitch must be 16 bytes)", what);
  if ((x_fmt == BSQ_NVFP4 || w_fmt == BSQ_NVFP4) && K % 32)
    return fail(BSQ_ERR_UNSUPPORTED, "%s: NVFP4 K %% 32 != 0 (packed row pitch must be 16 bytes)", what);
  if (M * N > 0 && (!y || !aligned16(y))) return fail(BSQ_ERR_INVALID_ARG, "%s: Y null or not 16-byte aligned", what);
  if (M == 0 || N == 0) return BSQ_OK;
  if (K == 0) return zero_output(y, M * N * 2, static_cast<cudaStream_t>(stream), what);
  int32_t* err = nullptr;
  int sms = 0;
  st = device_state(&err, &sms);
  if (st != BSQ_OK) return st;
  bsq::ForwardArgs a{x_fmt, w_fmt, x_data, x_scale, x_tensor_scale, w_data, w_scale, w_tensor_scale,
                     M, N, K, y, err, sms, static_cast<cudaStream_t>(stream)};
  const char* msg = "";
  if (bsq::launch_forward(a, &msg) != 0) return fail(BSQ_ERR_CUDA, "%s: %s", what, msg);
  return BSQ_OK;
}

bsq_status bsq_grouped_dgrad(const void* grad_out, int64_t S, int64_t N, int32_t w_fmt, const void* w_data,
                             const void* w_scale, const float* w_tensor_scale, int64_t E, int64_t K,
                             const int32_t* offsets, void* grad_x, void* stream) {
  const char* what = "bsq_grouped_dgrad";
  bsq_status st = check_gemm_common(what, grad_out, S, N, w_fmt, K, grad_x, S * K);
  if (st != BSQ_OK) return st;
  if (E < 1) return fail(BSQ_ERR_INVALID_ARG, "%s: E must be >= 1", what);
  if (E > bsq::kMaxExperts) return fail(BSQ_ERR_UNSUPPORTED, "%s: E > %d", what, bsq::kMaxExperts);
  if (!offsets) return fail(BSQ_ERR_INVALID_ARG, "%s: null offsets", what);
  st = check_packed(what, w_fmt, w_data, w_scale, w_tensor_scale, E, N, K, true);
  if (st != BSQ_OK) return st;
  if (S == 0 || K == 0) return BSQ_OK;
  if (N == 0) return fail(BSQ_ERR_UNSUPPORTED, "%s: N == 0 with S > 0 (rows to zero depend on offsets)", what);
  // A decode-sized call (S within the small-rows bound) is bound by reading the experts'
  // weights, not by the tensor cores: the small-M kernel computes every row.  Above the
  // bound the pair-tile GEMM does, less (when a tail bound is set) each expert's ragged
  // last tile of at most that many rows, which the small-M kernel then takes.  Both read
  // the same device offsets, so each row has exactly one owner.
  const bool packed_w = w_fmt != BSQ_BF16;
  int tail = 0;
  if (!packed_w || S > bsq::grouped_small_rows()) {
    tail = packed_w ? bsq::grouped_tail_rows() : 0;
    bsq::GemmArgs a{};
    a.op = bsq::kDgrad; a.fmt = w_fmt; a.p_data = w_data; a.p_scale = w_scale; a.p_tensor_scale = w_tensor_scale;
    a.p_batch = E; a.p_rows = N; a.kc = K; a.g = grad_out; a.S = S; a.N = N; a.offsets = offsets; a.E = E;
    a.out = grad_x; a.stream = static_cast<cudaStream_t>(stream); a.tail_rows = tail;
    st = run_gemm(a, what);
    if (st != BSQ_OK || tail == 0) return st;
  } else {
    tail = bsq::kTileN - 1;   // every expert here has fewer than kTileN rows: all of them
  }
  int32_t* err = nullptr;
  int sms = 0;
  st = device_state(&err, &sms);
  if (st != BSQ_OK) return st;
  bsq::SmallMArgs s{w_fmt, grad_out, w_data, w_scale, w_tensor_scale, S, N, K, grad_x, nullptr, sms,
                    static_cast<cudaStream_t>(stream), err, offsets, E, tail};
  const char* msg = "";
  if (bsq::launch_smallm_cluster(s, &msg) != 0) return fail(BSQ_ERR_CUDA, "%s: %s", what, msg);
  return BSQ_OK;
}

bsq_status bsq_grouped_wgrad(const void* grad_out, int64_t S, int64_t N, int32_t x_fmt, const void* x_data,
                             const void* x_scale, const float* x_tensor_scale, int64_t K, const int32_t* offsets,
                             int64_t E, void* grad_w, void* stream) {
  const char* what = "bsq_grouped_wgrad";
  bsq_status st = check_gemm_common(what, grad_out, S, N, x_fmt, K, grad_w, E * N * K);
  if (st != BSQ_OK) return st;
  if (E < 1) return fail(BSQ_ERR_INVALID_ARG, "%s: E must be >= 1", what);
  if (E > bsq::kMaxExperts) return fail(BSQ_ERR_UNSUPPORTED, "%s: E > %d", what, bsq::kMaxExperts);
  if (!offsets) return fail(BSQ_ERR_INVALID_ARG, "%s: null offsets", what);
  st = check_packed(what, x_fmt, x_data, x_scale, x_tensor_scale, 1, S, K, true);
  if (st != BSQ_OK) return st;
  if (N == 0 || K == 0) return BSQ_OK;
  if (S == 0) return zero_output(grad_w, E * N * K * 2, static_cast<cudaStream_t>(stream), what);
  bsq::GemmArgs a{};
  a.op = bsq::kWgrad; a.fmt = x_fmt; a.p_data = x_data; a.p_scale = x_scale; a.p_tensor_scale = x_tensor_scale;
  a.p_batch = 1; a.p_rows = S; a.kc = K; a.g = grad_out; a.S = S; a.N = N; a.offsets = offsets; a.E = E;
  a.out = grad_w; a.stream = static_cast<cudaStream_t>(stream);
  return run_gemm(a, what);
}

bsq_status bsq_quantize_e5m2(const void* g, int64_t n, int32_t margin, void* codes, void* deq, float* step,
                             float* amax, void* stream) {
  const char* what = "bsq_quantize_e5m2";
  if (n < 0) return fail(BSQ_ERR_INVALID_ARG, "%s: negative size", what);
  if (margin < 0 || margin > 30) return fail(BSQ_ERR_INVALID_ARG, "%s: margin %d outside 0..30", what, margin);
  if (!step || !amax || (reinterpret_cast<uintptr_t>(step) & 3u) || (reinterpret_cast<uintptr_t>(amax) & 3u))
    return fail(BSQ_ERR_INVALID_ARG, "%s: step and amax must be 4-byte aligned device words", what);
  if (n > 0 && (!g || !aligned16(g))) return fail(BSQ_ERR_INVALID_ARG, "%s: g null or not 16-byte aligned", what);
  if (n > 0 && (!codes || (reinterpret_cast<uintptr_t>(codes) & 7u)))
    return fail(BSQ_ERR_INVALID_ARG, "%s: codes null or not 8-byte aligned", what);
  if (deq && !aligned16(deq)) return fail(BSQ_ERR_INVALID_ARG, "%s: deq not 16-byte aligned", what);
  int32_t* err = nullptr;
  int sms = 0;
  bsq_status st = device_state(&err, &sms);
  if (st != BSQ_OK) return st;
  bsq::QuantArgs a{g, n, margin, codes, deq, step, amax, sms, static_cast<cudaStream_t>(stream)};
  const char* msg = "";
  if (bsq::launch_quantize_e5m2(a, &msg) != 0) return fail(BSQ_ERR_CUDA, "%s: %s", what, msg);
  return BSQ_OK;
}

bsq_status bsq_linear_backward_e5m2(const void* grad_out, int64_t M, int64_t N, int32_t w_fmt, const void* w_data,
                                    const void* w_scale, const float* w_tensor_scale, int32_t x_fmt,
                                    const void* x_data, const void* x_scale, const float* x_tensor_scale, int64_t K,
                                    uint32_t needs, int32_t margin, void* g_codes, void* g_deq, float* g_step,
                                    float* g_amax, void* grad_x, void* grad_w, void* stream) {
  const char* what = "bsq_linear_backward_e5m2";
  if (needs & ~static_cast<uint32_t>(BSQ_NEEDS_GRAD_X | BSQ_NEEDS_GRAD_W))
    return fail(BSQ_ERR_INVALID_ARG, "%s: unknown bits in needs (0x%x)", what, needs);
  if (M < 0 || N < 0) return fail(BSQ_ERR_INVALID_ARG, "%s: negative size", what);
  if (M * N > 0 && !g_deq) return fail(BSQ_ERR_INVALID_ARG, "%s: null g_deq", what);
  // the products' own checks come first, so that a bad operand launches nothing
  if (needs & BSQ_NEEDS_GRAD_X) {
    const bsq_status st = static_cast<bsq_status>(
        bsq::check_linear_dgrad_args(grad_out, M, N, w_fmt, w_data, w_scale, w_tensor_scale, K, grad_x));
    if (st != BSQ_OK) return st;
  }
  if (needs & BSQ_NEEDS_GRAD_W) {
    bsq_status st = check_gemm_common(what, grad_out, M, N, x_fmt, K, grad_w, N * K);
    if (st == BSQ_OK) st = check_packed(what, x_fmt, x_data, x_scale, x_tensor_scale, 1, M, K, true);
    if (st != BSQ_OK) return st;
  }
  bsq_status st = bsq_quantize_e5m2(grad_out, M * N, margin, g_codes, g_deq, g_step, g_amax, stream);
  if (st != BSQ_OK) return st;
  return bsq_linear_backward(g_deq, M, N, w_fmt, w_data, w_scale, w_tensor_scale, x_fmt, x_data, x_scale,
                             x_tensor_scale, K, needs, grad_x, grad_w, stream);
}

}  // extern "C"
