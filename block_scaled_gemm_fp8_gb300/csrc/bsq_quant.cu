// bsq_quant.cu -- per-tensor E5M2 quantization of a BF16 gradient, and E5M2 dequantization.
//
// AstrAI fp8.py, `_LinearFp8.backward` with the "hybrid" format: the backward quantizes the
// incoming gradient once to E5M2 and both products use that quantization.  The step of the
// tensor is (amax / 57344) / 2^margin, amax = max |g| in float32 clamped below at 1e-12
// (dynamic scaling: the current tensor's amax, `_dynamic_scale`).  Each element is divided
// by the step in float32 (IEEE division) and rounded to E5M2, ties to even, saturating to
// the finite range.  A dequantized copy, bf16(bf16(code) * bf16(step)) -- the library's
// dequantization rule -- can be written in the same pass.
//
// Two passes over the gradient, both bound by HBM: an amax reduction (four independent
// 16-byte loads in flight per thread, one atomic max per block on the float's bits, which
// order like the values for non-negative floats and put NaN above infinity), then the
// quantization (16-byte loads, 8-byte code stores, 16-byte stores of the dequantized copy).
//
// The quotient.  The code of an element is RN_e5m2(RN_f32(x / step)).  The quantization
// pass forms q1 = RN_f32(x * r) with r = RN_f32(1 / step) instead of dividing: q1 is within
// 3 float32 ulps of the IEEE quotient (two roundings of relative size 2^-24 each, the
// quotient's own half ulp, and up to a factor 2 from the position in the binade).  E5M2
// rounding is monotonic and changes only at the midpoints between neighbouring E5M2
// values, which in float32 are the numbers whose 23-bit mantissa has bit 20 set and bits
// 19..0 clear.  So when q1's low 21 mantissa bits are more than 4 away from that pattern,
// q1 and the quotient round to the same code; otherwise, and below 2^-13 (the E5M2
// subnormal range and its edge), the element takes the IEEE division.  Zeros, infinities
// and NaNs give the same codes either way (r is 0 when step is infinite, NaN when it is).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bsq_internal.h"
#include "../../include/bsq.h"

namespace bsq {

namespace {

constexpr int kQThreads = 256;
constexpr float kE5M2Max = 57344.0f;
constexpr float kAmaxFloor = 1e-12f;

// Larger of the two BF16 magnitudes of a pair (as 16-bit patterns: the order of the
// values, NaN patterns above infinity).
__device__ __forceinline__ uint32_t abs_max_pair(uint32_t w) {
  const uint32_t a = w & 0x7FFFu, b = (w >> 16) & 0x7FFFu;
  return a > b ? a : b;
}

__device__ __forceinline__ uint32_t abs_max_u4(const uint4& v) {
  return max(max(abs_max_pair(v.x), abs_max_pair(v.y)), max(abs_max_pair(v.z), abs_max_pair(v.w)));
}

__global__ void __launch_bounds__(kQThreads) amax_bf16_kernel(const uint4* __restrict__ g, int64_t n8,
                                                               const uint16_t* __restrict__ tail, int tail_n,
                                                               uint32_t* __restrict__ amax_bits) {
  uint32_t m = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kQThreads;
  int64_t i = static_cast<int64_t>(blockIdx.x) * kQThreads + threadIdx.x;
  for (; i + 3 * stride < n8; i += 4 * stride) {   // four loads in flight
    const uint4 a = __ldg(g + i), b = __ldg(g + i + stride), c = __ldg(g + i + 2 * stride), d = __ldg(g + i + 3 * stride);
    m = max(m, max(max(abs_max_u4(a), abs_max_u4(b)), max(abs_max_u4(c), abs_max_u4(d))));
  }
  for (; i < n8; i += stride) m = max(m, abs_max_u4(__ldg(g + i)));
  if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < tail_n) m = max(m, static_cast<uint32_t>(tail[threadIdx.x] & 0x7FFFu));
  m = __reduce_max_sync(0xffffffffu, m);
  __shared__ uint32_t wm[kQThreads / 32];
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < kQThreads / 32 ? wm[threadIdx.x] : 0u;
    m = __reduce_max_sync(0xffffffffu, m);
    if (threadIdx.x == 0 && m) atomicMax(amax_bits, m << 16);   // BF16 pattern -> float32 pattern
  }
}

// float32 values of the step and amax from the reduced amax bits (NaN stays NaN).
__device__ __forceinline__ float amax_of(uint32_t bits) {
  const float a = __uint_as_float(bits);
  return isnan(a) ? a : fmaxf(a, kAmaxFloor);
}

// Two float32 values -> two E5M2 codes (lo in bits 0-7, hi in bits 8-15): RN, saturating.
__device__ __forceinline__ uint32_t e5m2x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// Two E5M2 codes (bits 0-7, 8-15 of c) times the BF16 step s -> a BF16 pair, one rounding.
__device__ __forceinline__ uint32_t e5m2x2_dequant(uint32_t c, float s) {
  // each code is the high byte of an FP16 number with the same value
  const uint32_t h = ((c & 0xFFu) << 8) | ((c & 0xFF00u) << 16);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  const __nv_bfloat162 r = __floats2bfloat162_rn(f.x * s, f.y * s);   // exact products
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ float bf16_round_f(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// RN_f32(x / step), from q1 = x * rcp where that gives the same E5M2 code (see the top of
// the file), else from the IEEE division.
__device__ __forceinline__ float e5m2_quotient(float x, float step, float rcp) {
  const float q = x * rcp;
  const uint32_t u = __float_as_uint(q) & 0x7FFFFFFFu;
  const uint32_t low = u & 0x1FFFFFu;
  const bool near_mid = low - 0xFFFFCu <= 8u;         // |low - 0x100000| <= 4
  const bool small = u < 0x39000000u && u != 0u;      // 0 < |q1| < 2^-13
  return (near_mid || small) ? __fdiv_rn(x, step) : q;
}

__global__ void __launch_bounds__(kQThreads) quantize_e5m2_kernel(const uint4* __restrict__ g, int64_t n8,
                                                                   const uint16_t* __restrict__ g_tail, int tail_n,
                                                                   uint32_t* __restrict__ amax_bits, int margin,
                                                                   uint2* __restrict__ codes, uint8_t* __restrict__ codes_tail,
                                                                   uint4* __restrict__ deq, uint16_t* __restrict__ deq_tail,
                                                                   float* __restrict__ step_out) {
  const float amax = amax_of(*reinterpret_cast<volatile uint32_t*>(amax_bits));
  const float step = __fdiv_rn(__fdiv_rn(amax, kE5M2Max), __int_as_float((127 + margin) << 23));   // margin 0..30
  const float rcp = __frcp_rn(step);
  const float s_bf = bf16_round_f(step);
  // eight elements at index i: codes, and the dequantized copy when asked for
  auto put = [&](const uint4& v, int64_t i) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t c2[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      c2[j] = e5m2x2(e5m2_quotient(__uint_as_float(w[j] << 16), step, rcp),
                     e5m2_quotient(__uint_as_float(w[j] & 0xFFFF0000u), step, rcp));
    codes[i] = make_uint2(c2[0] | (c2[1] << 16), c2[2] | (c2[3] << 16));
    if (deq)
      deq[i] = make_uint4(e5m2x2_dequant(c2[0], s_bf), e5m2x2_dequant(c2[1], s_bf), e5m2x2_dequant(c2[2], s_bf),
                          e5m2x2_dequant(c2[3], s_bf));
  };
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kQThreads;
  int64_t i = static_cast<int64_t>(blockIdx.x) * kQThreads + threadIdx.x;
  for (; i + 3 * stride < n8; i += 4 * stride) {   // four loads in flight
    const uint4 a = __ldg(g + i), b = __ldg(g + i + stride), c = __ldg(g + i + 2 * stride), d = __ldg(g + i + 3 * stride);
    put(a, i);
    put(b, i + stride);
    put(c, i + 2 * stride);
    put(d, i + 3 * stride);
  }
  for (; i < n8; i += stride) put(__ldg(g + i), i);
  if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < tail_n) {
    const float x = __uint_as_float(static_cast<uint32_t>(g_tail[threadIdx.x]) << 16);
    const uint32_t c = e5m2x2(__fdiv_rn(x, step), 0.f) & 0xFFu;
    codes_tail[threadIdx.x] = static_cast<uint8_t>(c);
    if (deq_tail) deq_tail[threadIdx.x] = static_cast<uint16_t>(e5m2x2_dequant(c, s_bf) & 0xFFFFu);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    step_out[0] = step;
    // the clamped amax replaces the reduced bits; a block still reading them derives the
    // same value from either (the clamp is idempotent)
    *reinterpret_cast<volatile float*>(amax_bits) = amax;
  }
}

// E5M2 codes with one float32 step per batch entry -> BF16 (8 elements per thread step).
__global__ void __launch_bounds__(kQThreads) dequant_e5m2_kernel(const uint2* __restrict__ codes, int64_t n8,
                                                                  int64_t units_per_batch, const float* __restrict__ steps,
                                                                  uint4* __restrict__ out) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kQThreads + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * kQThreads) {
    const uint2 c = __ldg(codes + i);
    const float s = bf16_round_f(__ldg(steps + i / units_per_batch));
    out[i] = make_uint4(e5m2x2_dequant(c.x & 0xFFFFu, s), e5m2x2_dequant(c.x >> 16, s),
                        e5m2x2_dequant(c.y & 0xFFFFu, s), e5m2x2_dequant(c.y >> 16, s));
  }
}

}  // namespace

int launch_quantize_e5m2(const QuantArgs& a, const char** msg) {
  const int64_t n8 = a.n / 8;
  const int tail = static_cast<int>(a.n % 8);
  // four resident blocks of 256 threads per SM, each thread with four 16-byte loads in flight
  int64_t blocks = (n8 + 4 * kQThreads - 1) / (4 * kQThreads);
  const int64_t cap = static_cast<int64_t>(a.num_sms) * 4;
  blocks = blocks < 1 ? 1 : (blocks > cap ? cap : blocks);
  const uint16_t* g16 = static_cast<const uint16_t*>(a.g);
  uint8_t* c8 = static_cast<uint8_t*>(a.codes);
  uint16_t* d16 = static_cast<uint16_t*>(a.deq);
  uint32_t* amax_bits = reinterpret_cast<uint32_t*>(a.amax);
  cudaError_t e = cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t), a.stream);
  if (e == cudaSuccess) {
    amax_bf16_kernel<<<static_cast<unsigned>(blocks), kQThreads, 0, a.stream>>>(
        static_cast<const uint4*>(a.g), n8, g16 + n8 * 8, tail, amax_bits);
    quantize_e5m2_kernel<<<static_cast<unsigned>(blocks), kQThreads, 0, a.stream>>>(
        static_cast<const uint4*>(a.g), n8, g16 + n8 * 8, tail, amax_bits, a.margin, static_cast<uint2*>(a.codes),
        c8 + n8 * 8, static_cast<uint4*>(a.deq), d16 ? d16 + n8 * 8 : nullptr, a.step);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    *msg = cudaGetErrorString(e);
    return static_cast<int>(e);
  }
  return 0;
}

int launch_dequant_e5m2(const DequantArgs& a, const char** msg) {
  const int64_t n8 = a.batch * a.rows * a.cols / 8;   // cols % 16 == 0
  if (n8 == 0) return 0;
  int64_t blocks = (n8 + kQThreads - 1) / kQThreads;
  const int64_t cap = static_cast<int64_t>(a.num_sms) * 8;
  if (blocks > cap) blocks = cap;
  dequant_e5m2_kernel<<<static_cast<unsigned>(blocks), kQThreads, 0, a.stream>>>(
      static_cast<const uint2*>(a.data), n8, a.rows * a.cols / 8, static_cast<const float*>(a.scale),
      static_cast<uint4*>(a.out));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *msg = cudaGetErrorString(e);
    return static_cast<int>(e);
  }
  return 0;
}

}  // namespace bsq
