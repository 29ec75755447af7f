// bsq_smallm.cu -- dgrad for a handful of token rows (M <= 16): grad_X[M,K] = grad_out[M,N] @ deq(W)[N,K]
// (MSLK PR #393 "Implementation Method"; transformers PR #50031 `FP8LinearFunction.backward`).
//
// With M this small the product is bound by reading the packed weight once from HBM, so
// the kernel is shaped for bandwidth, not for the tensor-core peak:
//   * split-K over the N rows of W: every CTA owns a 128-column slab of K and a range of
//     rows, so the whole GPU streams W concurrently (two CTAs per SM);
//   * the packed bytes go straight from global memory into registers (64-byte contiguous
//     row segments per load instruction) and are decoded there -- no shared-memory staging
//     of the BF16 weight;
//   * decoding pairs the same column of two adjacent rows in one 32-bit register
//     (one byte permute + the multiply-spread of bsq_decode.cuh), which is exactly the
//     k-pair an mma.sync B fragment wants, so no transpose is needed;
//   * m16n8k16 BF16 mma.sync with FP32 accumulators (tokens are the M=16 side);
//   * the CTAs of a slab reduce through an FP32 workspace with atomics; the last CTA to
//     finish a slab converts it to BF16, writes grad_X and zeroes the workspace again.
#include <cstdio>
#include <mutex>

#include <cuda_bf16.h>

#include "bsq_decode.cuh"
#include "bsq_internal.h"
#include "../../include/bsq.h"

namespace bsq {

namespace {

constexpr int kWarps = 8;
constexpr int kThreadsSm = kWarps * 32;
constexpr int kSlab = 128;       // columns of K per CTA
constexpr int kStep = 16;        // rows of N per mma k-step
constexpr int kNT = 16;          // n-tiles (8 columns each) per warp per k-step

struct SmallParams {
  const __nv_bfloat16* g;
  const uint8_t* w;
  const uint8_t* scale;
  const float* tensor_scale;
  __nv_bfloat16* out;
  float* ws;          // [16][K] FP32, all zero between calls
  int32_t* counters;  // [num_slabs], all zero between calls
  int32_t M, N, K;
  int32_t rows_per_split;
  int32_t scale_ld;   // MXFP4: K/32, NVFP4: K/16, FP8: ceil(K/128)
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Scale pair for two rows: (s_a, s_b) with the combined fast path only when both are exact.
__device__ __forceinline__ ScaleBf16 pair_scales(const ScaleBf16& a, const ScaleBf16& b) {
  ScaleBf16 r;
  r.s2 = (a.s2 & 0xFFFFu) | (b.s2 & 0xFFFF0000u);
  r.c2 = (a.c2 & 0xFFFFu) | (b.c2 & 0xFFFF0000u);
  r.fast = a.fast && b.fast;
  return r;
}

__device__ __forceinline__ uint32_t scale_one(uint32_t v, const ScaleBf16& s, uint32_t pow2k_x2) {
  return s.fast ? bf16x2_mul(v, s.c2) : bf16x2_mul(bf16x2_mul(v, pow2k_x2), s.s2);
}

// Byte `b` (0..3) of word x in the low half and of word y in the high half.
__device__ __forceinline__ uint32_t pair_bytes(uint32_t x, uint32_t y, int b) {
  return prmt(x, y, static_cast<uint32_t>(b | (b << 4) | ((4 + b) << 8) | ((4 + b) << 12)));
}

template <int FMT>
struct RowData;  // packed bytes of one thread's 16 columns in one row

template <>
struct RowData<BSQ_MXFP4> { uint2 v; };
template <>
struct RowData<BSQ_NVFP4> { uint2 v; };
template <>
struct RowData<BSQ_FP8_E4M3_B128> { uint4 v; };

template <int FMT>
__device__ __forceinline__ void load_row(RowData<FMT>& d, const SmallParams& p, int row, int col, bool ok) {
  if (FMT == BSQ_FP8_E4M3_B128) {
    uint4 z = make_uint4(0, 0, 0, 0);
    if (ok) z = __ldg(reinterpret_cast<const uint4*>(p.w + static_cast<int64_t>(row) * p.K + col));
    reinterpret_cast<uint4&>(d.v) = z;
  } else {
    uint2 z = make_uint2(0, 0);
    if (ok) z = __ldg(reinterpret_cast<const uint2*>(p.w + static_cast<int64_t>(row) * (p.K / 2) + col / 2));
    reinterpret_cast<uint2&>(d.v) = z;
  }
}

// One k-step worth of raw inputs of this thread: rows (a,b) feed B register 0, rows (c,d) register 1.
template <int FMT>
struct StepData {
  RowData<FMT> r[4];
  uint32_t sraw[4];   // FP4: scale byte per row
  float sf;           // FP8: block scale (all four rows share one 128-row block)
};

template <int FMT>
__device__ __forceinline__ void load_step(StepData<FMT>& s, const SmallParams& p, int base, int q, int col,
                                          bool col_ok, int n1) {
  const int rows[4] = {base + 2 * q, base + 2 * q + 1, base + 8 + 2 * q, base + 9 + 2 * q};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool ok = col_ok && rows[i] < n1;
    load_row<FMT>(s.r[i], p, rows[i], col, ok);
    s.sraw[i] = 0;
    if (FMT == BSQ_MXFP4 && ok) s.sraw[i] = __ldg(p.scale + static_cast<int64_t>(rows[i]) * p.scale_ld + (col >> 5));
    if (FMT == BSQ_NVFP4 && ok) s.sraw[i] = __ldg(p.scale + static_cast<int64_t>(rows[i]) * p.scale_ld + (col >> 4));
  }
  s.sf = 0.f;
  if (FMT == BSQ_FP8_E4M3_B128 && col_ok && base < n1)
    s.sf = __ldg(reinterpret_cast<const float*>(p.scale) + static_cast<int64_t>(base >> 7) * p.scale_ld + (col >> 7));
}

template <int FMT>
__device__ __forceinline__ ScaleBf16 row_scale(uint32_t raw, float tscale) {
  if (FMT == BSQ_MXFP4) return make_scale_e8m0(raw);
  return make_scale_nvfp4(raw, tscale);
}

// Decode part `wi` of one k-step into B fragments for n-tiles [kPart*wi, kPart*(wi+1)):
// b0[i] from rows (a,b), b1[i] from rows (c,d).  FP4: 2 parts of 8 n-tiles (one packed
// word per row each); FP8: 4 parts of 4 n-tiles.
template <int FMT>
struct Part {
  static constexpr int kParts = FMT == BSQ_FP8_E4M3_B128 ? 4 : 2;
  static constexpr int kTiles = kNT / kParts;
};

template <int FMT>
__device__ __forceinline__ void decode_part(const StepData<FMT>& s, float tscale, int wi,
                                            uint32_t (&b0)[Part<FMT>::kTiles], uint32_t (&b1)[Part<FMT>::kTiles]) {
  if (FMT == BSQ_FP8_E4M3_B128) {
    const ScaleBf16 sc = make_scale_fp8(s.sf);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const uint32_t* xw = reinterpret_cast<const uint32_t*>(&s.r[2 * half].v);
      const uint32_t* yw = reinterpret_cast<const uint32_t*>(&s.r[2 * half + 1].v);
      uint32_t(&dst)[Part<FMT>::kTiles] = half ? b1 : b0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t v = pair_bytes(xw[wi], yw[wi], j);   // column 4wi+j of both rows
        uint32_t o = scale_one(((v << 4) & 0x07F007F0u) | ((v << 8) & 0x80008000u), sc, kPow2_120x2);
        if ((v & 0x7Fu) == 0x7Fu) o = (o & 0xFFFF0000u) | kBf16NaN;             // E4M3 NaN, first row
        if ((v & 0x007F0000u) == 0x007F0000u) o = (o & 0xFFFFu) | (kBf16NaN << 16);  // second row
        dst[j] = o;
      }
    }
  } else {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const uint32_t* xw = reinterpret_cast<const uint32_t*>(&s.r[2 * half].v);
      const uint32_t* yw = reinterpret_cast<const uint32_t*>(&s.r[2 * half + 1].v);
      const ScaleBf16 sc = pair_scales(row_scale<FMT>(s.sraw[2 * half], tscale),
                                       row_scale<FMT>(s.sraw[2 * half + 1], tscale));
      uint32_t(&dst)[Part<FMT>::kTiles] = half ? b1 : b0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t v = pair_bytes(xw[wi], yw[wi], j);          // byte 4wi+j of both rows
        const uint32_t lo = ((v & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;   // column 8wi+2j
        const uint32_t hi = ((v & 0x00F000F0u) * 0x0104u) & 0x81C081C0u;   // column 8wi+2j+1
        dst[2 * j] = scale_one(lo, sc, kPow2_126x2);
        dst[2 * j + 1] = scale_one(hi, sc, kPow2_126x2);
      }
    }
  }
}

template <int FMT>
__global__ void __launch_bounds__(kThreadsSm, 2) smallm_dgrad_kernel(const SmallParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int slab = blockIdx.x;
  const int cb = slab * kSlab;
  const int n0 = blockIdx.y * p.rows_per_split;
  const int n1 = min(p.N, n0 + p.rows_per_split);
  const int nrows = max(n1 - n0, 0);
  const int pitch = p.rows_per_split + 8;   // bf16 elements per token row of the G slab (16-byte skew)
  __nv_bfloat16* gs = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  float* red = reinterpret_cast<float*>(smem_raw + static_cast<size_t>(16) * pitch * 2);
  __shared__ int last_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;

  // grad_out slab [16 tokens][rows] (zero past M or past the row range) and the reduction buffer
  for (int i = tid; i < 16 * (pitch / 2); i += kThreadsSm) {
    const int t = i / (pitch / 2), c2 = (i % (pitch / 2)) * 2;
    uint32_t v = 0;
    if (t < p.M && c2 < nrows)  // nrows is even: N % 8 == 0 and n0 % 16 == 0
      v = __ldg(reinterpret_cast<const uint32_t*>(p.g + static_cast<int64_t>(t) * p.N + n0 + c2));
    reinterpret_cast<uint32_t*>(gs)[t * (pitch / 2) + c2 / 2] = v;
  }
  __syncthreads();

  float tscale = 0.f;
  if (FMT == BSQ_NVFP4) tscale = __ldg(p.tensor_scale);
  const int col = cb + 16 * g;
  const bool col_ok = col < p.K;
  float acc[kNT][4];
#pragma unroll
  for (int i = 0; i < kNT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  const int nsteps = (nrows + kStep - 1) / kStep;
  StepData<FMT> cur, nxt;
  int ks = warp;
  if (ks < nsteps) load_step<FMT>(cur, p, n0 + ks * kStep, q, col, col_ok, n1);
  for (; ks < nsteps; ks += kWarps) {
    const int ks2 = ks + kWarps;
    if (ks2 < nsteps) load_step<FMT>(nxt, p, n0 + ks2 * kStep, q, col, col_ok, n1);
    // A fragment: grad_out[token][k] for k = local rows ks*16 .. +15
    const uint32_t* g32 = reinterpret_cast<const uint32_t*>(gs);
    const int k0 = ks * kStep;
    uint32_t a[4];
    a[0] = g32[g * (pitch / 2) + (k0 + 2 * q) / 2];
    a[1] = g32[(g + 8) * (pitch / 2) + (k0 + 2 * q) / 2];
    a[2] = g32[g * (pitch / 2) + (k0 + 8 + 2 * q) / 2];
    a[3] = g32[(g + 8) * (pitch / 2) + (k0 + 8 + 2 * q) / 2];
#pragma unroll
    for (int wi = 0; wi < Part<FMT>::kParts; ++wi) {
      uint32_t b0[Part<FMT>::kTiles], b1[Part<FMT>::kTiles];
      decode_part<FMT>(cur, tscale, wi, b0, b1);
#pragma unroll
      for (int i = 0; i < Part<FMT>::kTiles; ++i) mma_bf16_16816(acc[wi * Part<FMT>::kTiles + i], a, b0[i], b1[i]);
    }
    if (ks2 < nsteps) cur = nxt;
  }

  // Cross-warp reduction through per-warp slabs laid out [nt][token][n] (8-byte stores of
  // fragment column pairs, no bank conflicts); fragment column n of n-tile nt is output
  // column cb + 16 n + nt.
  {
    float* mine = red + warp * (kNT * 16 * 8);
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      *reinterpret_cast<float2*>(mine + (nt * 16 + g) * 8 + 2 * q) = make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2*>(mine + (nt * 16 + g + 8) * 8 + 2 * q) = make_float2(acc[nt][2], acc[nt][3]);
    }
  }
  __syncthreads();
  // thread i sums the 8 warps for slab entries i, i + 256, ... (entry = (nt, token, n))
  for (int i = tid; i < kNT * 16 * 8; i += kThreadsSm) {
    float v = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) v += red[w2 * (kNT * 16 * 8) + i];
    red[kWarps * (kNT * 16 * 8) + i] = v;
  }
  __syncthreads();
  red += kWarps * (kNT * 16 * 8);   // reduced slab, same layout
  // entry i = (nt, token t, fragment column n) holds output (t, cb + 16 n + nt); walking
  // i = t*128 + c_local order keeps the global accesses coalesced.
  auto entry = [](int t, int cl) { return ((cl & 15) * 16 + t) * 8 + (cl >> 4); };
  if (gridDim.y == 1) {
    for (int i = tid; i < 16 * kSlab; i += kThreadsSm) {
      const int t = i / kSlab, cl = i % kSlab, c = cb + cl;
      if (t < p.M && c < p.K) p.out[static_cast<int64_t>(t) * p.K + c] = __float2bfloat16_rn(red[entry(t, cl)]);
    }
    return;
  }
  for (int i = tid; i < 16 * kSlab; i += kThreadsSm) {
    const int t = i / kSlab, cl = i % kSlab, c = cb + cl;
    if (t < p.M && c < p.K) atomicAdd(p.ws + static_cast<int64_t>(t) * p.K + c, red[entry(t, cl)]);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) last_flag = (atomicAdd(p.counters + slab, 1) == static_cast<int>(gridDim.y) - 1);
  __syncthreads();
  if (!last_flag) return;
  __threadfence();
  for (int i = tid; i < 16 * kSlab; i += kThreadsSm) {
    const int t = i / kSlab, c = cb + i % kSlab;
    if (t < p.M && c < p.K) {
      float* w = p.ws + static_cast<int64_t>(t) * p.K + c;
      p.out[static_cast<int64_t>(t) * p.K + c] = __float2bfloat16_rn(__ldcg(w));
      __stcg(w, 0.f);
    }
  }
  if (tid == 0) p.counters[slab] = 0;
}

}  // namespace

size_t smallm_workspace_bytes(int64_t K) {
  const int64_t slabs = (K + kSlab - 1) / kSlab;
  return static_cast<size_t>(16 * K * 4 + ((slabs * 4 + 255) / 256) * 256 + 256);
}

int launch_smallm(const SmallMArgs& a, const char** msg) {
  SmallParams p;
  p.g = static_cast<const __nv_bfloat16*>(a.g);
  p.w = static_cast<const uint8_t*>(a.w_data);
  p.scale = static_cast<const uint8_t*>(a.w_scale);
  p.tensor_scale = a.w_tensor_scale;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.M = static_cast<int32_t>(a.M);
  p.N = static_cast<int32_t>(a.N);
  p.K = static_cast<int32_t>(a.K);
  p.scale_ld = a.fmt == BSQ_MXFP4 ? static_cast<int32_t>(a.K / 32)
               : a.fmt == BSQ_NVFP4 ? static_cast<int32_t>(a.K / 16)
                                    : static_cast<int32_t>((a.K + 127) / 128);
  const int slabs = static_cast<int>((a.K + kSlab - 1) / kSlab);
  // about two CTAs per SM in one wave, at most 1024 rows of W per CTA
  int splits = (2 * a.num_sms + slabs - 1) / slabs;
  splits = splits < 1 ? 1 : splits;
  int rps = static_cast<int>((a.N + splits - 1) / splits);
  rps = (rps + kStep - 1) / kStep * kStep;
  if (rps > 1024) rps = 1024;
  if (rps < kStep) rps = kStep;
  splits = static_cast<int>((a.N + rps - 1) / rps);
  p.rows_per_split = rps;
  p.ws = static_cast<float*>(a.ws);
  p.counters = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(a.ws) + static_cast<size_t>(16 * a.K * 4));
  if (splits > 1 && !a.ws) {
    *msg = "small-M dgrad needs a workspace";
    return -1;
  }
  const size_t smem = static_cast<size_t>(16) * (rps + 8) * 2 + (kWarps + 1) * kNT * 16 * 8 * 4;
  const dim3 grid(slabs, splits);
  cudaError_t e = cudaSuccess;
  switch (a.fmt) {
    case BSQ_MXFP4:
      e = cudaFuncSetAttribute(smallm_dgrad_kernel<BSQ_MXFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e == cudaSuccess) smallm_dgrad_kernel<BSQ_MXFP4><<<grid, kThreadsSm, smem, a.stream>>>(p);
      break;
    case BSQ_NVFP4:
      e = cudaFuncSetAttribute(smallm_dgrad_kernel<BSQ_NVFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e == cudaSuccess) smallm_dgrad_kernel<BSQ_NVFP4><<<grid, kThreadsSm, smem, a.stream>>>(p);
      break;
    case BSQ_FP8_E4M3_B128:
      e = cudaFuncSetAttribute(smallm_dgrad_kernel<BSQ_FP8_E4M3_B128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e == cudaSuccess) smallm_dgrad_kernel<BSQ_FP8_E4M3_B128><<<grid, kThreadsSm, smem, a.stream>>>(p);
      break;
    default:
      *msg = "small-M dgrad: unsupported format";
      return -1;
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    *msg = cudaGetErrorString(e);
    return static_cast<int>(e);
  }
  return 0;
}

}  // namespace bsq

// ---------------------------------------------------------------- allocation-free entry point
// Some callers cannot call cudaMalloc at all: code running inside a CUDA graph that is being
// captured, allocators that own every byte of device memory, or hosts that forbid device
// allocation after start-up.  bsq_linear_dgrad_smallm_noalloc serves them with the small-M
// kernel above, its split-K scratch living in this file-scope device array instead of the
// lazily allocated workspace.  The array exists on every device that loads the library,
// for the life of the process.
namespace {

constexpr int64_t kStaticMaxK = 16384;  // largest K the static scratch serves
constexpr size_t kStaticScratchBytes = 16 * kStaticMaxK * 4 + 4096;
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevicesStatic = 64;
void* g_static_ptr[kMaxDevicesStatic] = {};
int g_static_sms[kMaxDevicesStatic] = {};
std::mutex g_static_mu;

}  // namespace

extern "C" bsq_status bsq_linear_dgrad_smallm_noalloc(const void* grad_out, int64_t M, int64_t N, int32_t w_fmt,
                                                      const void* w_data, const void* w_scale,
                                                      const float* w_tensor_scale, int64_t K, void* grad_x,
                                                      void* stream) {
  const int st = bsq::check_linear_dgrad_args(grad_out, M, N, w_fmt, w_data, w_scale, w_tensor_scale, K, grad_x);
  if (st != BSQ_OK) return static_cast<bsq_status>(st);
  if (M > bsq::kSmallM)
    return static_cast<bsq_status>(
        bsq::set_error(BSQ_ERR_UNSUPPORTED, "bsq_linear_dgrad_smallm_noalloc: M must be <= 16"));
  if (w_fmt == BSQ_BF16)
    return static_cast<bsq_status>(
        bsq::set_error(BSQ_ERR_UNSUPPORTED, "bsq_linear_dgrad_smallm_noalloc: W must be FP8, MXFP4 or NVFP4"));
  if (K > kStaticMaxK || bsq::smallm_workspace_bytes(K) > kStaticScratchBytes)
    return static_cast<bsq_status>(bsq::set_error(
        BSQ_ERR_UNSUPPORTED, "bsq_linear_dgrad_smallm_noalloc: K exceeds the static scratch maximum of 16384"));
  if (M == 0 || K == 0) return BSQ_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (N == 0) {
    const cudaError_t e = cudaMemsetAsync(grad_x, 0, static_cast<size_t>(M * K * 2), s);
    return e == cudaSuccess ? BSQ_OK
                            : static_cast<bsq_status>(bsq::set_error(BSQ_ERR_CUDA, cudaGetErrorString(e)));
  }
  // Per-device set-up on the first call (device current): the array's device address.
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevicesStatic)
    return static_cast<bsq_status>(bsq::set_error(BSQ_ERR_CUDA, "bsq_linear_dgrad_smallm_noalloc: no device"));
  void* scratch = nullptr;
  int sms = 0;
  {
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev]) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_static_scratch);
      if (e != cudaSuccess)
        return static_cast<bsq_status>(bsq::set_error(BSQ_ERR_CUDA, cudaGetErrorString(e)));
      int n = 0;
      e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess)
        return static_cast<bsq_status>(bsq::set_error(BSQ_ERR_CUDA, cudaGetErrorString(e)));
      g_static_ptr[dev] = ptr;
      g_static_sms[dev] = n;
    }
    scratch = g_static_ptr[dev];
    sms = g_static_sms[dev];
  }
  // The kernel needs the scratch at zero on entry (and leaves it so); clear the part this
  // call uses so that an earlier interrupted call cannot leak into this one.
  e = cudaMemsetAsync(scratch, 0, bsq::smallm_workspace_bytes(K), s);
  if (e != cudaSuccess) return static_cast<bsq_status>(bsq::set_error(BSQ_ERR_CUDA, cudaGetErrorString(e)));
  bsq::SmallMArgs a{w_fmt, grad_out, w_data, w_scale, w_tensor_scale, M, N, K, grad_x, scratch, sms, s};
  const char* msg = "";
  if (bsq::launch_smallm(a, &msg) != 0) return static_cast<bsq_status>(bsq::set_error(BSQ_ERR_CUDA, msg));
  return BSQ_OK;
}

