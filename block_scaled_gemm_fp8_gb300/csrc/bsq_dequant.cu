// bsq_dequant.cu -- standalone dequantization of a packed operand to BF16 in HBM.
//
// The operation is the backward's "dequantize to BF16" step on its own
// (transformers PR #50031 `_dequantize_fp8_weight`; MSLK PR #393's FP4 dequantization
// helpers), used when a BF16 copy is wanted or as the first half of the
// dequantize-then-multiply path.  It is bound by HBM bandwidth.
//   FP4: every lane reads 4-byte words of 8 codes, eight per step, so each warp load reads
//        128 contiguous bytes and each 16-byte store instruction writes 512 contiguous
//        bytes of BF16.  (16-byte loads of 32 codes per lane leave each lane a 64-byte run
//        of output, so every store instruction scatters half sectors: measured at about
//        half the bandwidth.)  Scales: one E8M0 / E4M3 byte per 8 codes.
//   FP8: every lane reads 16-byte loads of 16 codes of one row (two in flight) and writes
//        two 16-byte stores; one scale_inv per load (a load never crosses a 128-column
//        scale block), its index formed once per 16 codes.
#include <cuda_bf16.h>

#include "bsq_decode.cuh"
#include "bsq_internal.h"
#include "../../include/bsq.h"

namespace bsq {

namespace {

constexpr int kThreads = 256;
constexpr int kWordsPerLane = 8;   // FP4: 8 words (32 bytes) of codes in flight per lane

// MXFP4 / NVFP4: one 32-bit word = 8 codes = 16 output bytes.
template <int FMT>
__global__ void __launch_bounds__(kThreads) dequant_fp4_kernel(const uint32_t* __restrict__ data,
                                                               const uint8_t* __restrict__ scale,
                                                               const float* __restrict__ tscale, int64_t n_words,
                                                               int64_t words_per_batch, uint4* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  constexpr int64_t kWarpWords = 32 * kWordsPerLane;
  // NVFP4 with one tensor scale for the whole launch: the combined scale of each of the 256
  // E4M3 block codes, built once per CTA (thread t: code t), fast flags as a bit mask.
  __shared__ uint2 lut[FMT == BSQ_NVFP4 ? 256 : 1];
  __shared__ uint32_t lut_fast[FMT == BSQ_NVFP4 ? 8 : 1];
  const bool one_ts = FMT == BSQ_NVFP4 && words_per_batch >= n_words;
  if (one_ts) {
    static_assert(FMT != BSQ_NVFP4 || kThreads == 256, "one table entry per thread");
    const ScaleBf16 c = make_scale_nvfp4(threadIdx.x, __ldg(tscale));
    lut[threadIdx.x] = make_uint2(c.s2, c.c2);
    const uint32_t fast = __ballot_sync(0xffffffffu, c.fast);
    if (lane == 0) lut_fast[threadIdx.x >> 5] = fast;
    __syncthreads();
  }
  for (int64_t base = warp * kWarpWords; base < n_words; base += nwarps * kWarpWords) {
    uint32_t w[kWordsPerLane];
    uint32_t sb[kWordsPerLane];
#pragma unroll
    for (int j = 0; j < kWordsPerLane; ++j) {
      const int64_t idx = base + lane + 32 * j;
      w[j] = 0;
      sb[j] = 0;
      if (idx < n_words) {
        w[j] = __ldg(data + idx);
        sb[j] = __ldg(scale + (FMT == BSQ_MXFP4 ? (idx >> 2) : (idx >> 1)));
      }
    }
#pragma unroll
    for (int j = 0; j < kWordsPerLane; ++j) {
      const int64_t idx = base + lane + 32 * j;
      if (idx >= n_words) continue;
      ScaleBf16 s;
      if (FMT == BSQ_MXFP4) {
        s = make_scale_e8m0(sb[j]);
      } else {
        if (one_ts) {
          const uint2 c = lut[sb[j]];
          s.s2 = c.x;
          s.c2 = c.y;
          s.fast = (lut_fast[sb[j] >> 5] >> (sb[j] & 31u)) & 1u;
        } else {
          s = make_scale_nvfp4(sb[j], __ldg(tscale + idx / words_per_batch));
        }
      }
      uint32_t p[4];
      decode_e2m1x8(w[j], s, p);
      uint4 o;
      unzip_pairs(p[0], p[1], o.x, o.z);  // (c0,c1), (c4,c5)
      unzip_pairs(p[2], p[3], o.y, o.w);  // (c2,c3), (c6,c7)
      out[idx] = o;
    }
  }
}

// FP8 E4M3, 16-byte form: one uint4 = 16 codes of one row (cols % 16 == 0, so a load never
// crosses a row or a 128-column scale block) = 2 output uint4, two loads in flight.
__global__ void __launch_bounds__(kThreads) dequant_fp8_x2_kernel(const uint4* __restrict__ data,
                                                                  const float* __restrict__ scale_inv,
                                                                  int64_t n_pairs, int64_t rows, int64_t cols,
                                                                  int shift, uint4* __restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  const int64_t per_row = cols >> 4;
  const int64_t rblocks = shift >= 31 ? 1 : (rows + (1 << shift) - 1) >> shift;
  const int64_t cblocks = shift >= 31 ? 1 : (cols + (1 << shift) - 1) >> shift;
  auto scale_of = [&](int64_t i) {
    const int64_t grow = i / per_row;               // row across the whole batch
    const int64_t col = (i - grow * per_row) << 4;
    const int64_t b = grow / rows;
    const int64_t r = grow - b * rows;
    return __ldg(scale_inv + (b * rblocks + (r >> shift)) * cblocks + (col >> shift));
  };
  auto put = [&](const uint4& w, float sv, int64_t i) {
    const ScaleBf16 s = make_scale_fp8(sv);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t a02, a13, b02, b13;
      decode_e4m3x4(ws[2 * h], s, a02, a13);
      decode_e4m3x4(ws[2 * h + 1], s, b02, b13);
      uint4 o;
      unzip_pairs(a02, a13, o.x, o.y);  // (c0,c1), (c2,c3)
      unzip_pairs(b02, b13, o.z, o.w);  // (c4,c5), (c6,c7)
      out[2 * i + h] = o;
    }
  };
  int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  for (; i + stride < n_pairs; i += 2 * stride) {
    const uint4 wa = __ldg(data + i), wb = __ldg(data + i + stride);
    const float sa = scale_of(i), sb = scale_of(i + stride);
    put(wa, sa, i);
    put(wb, sb, i + stride);
  }
  if (i < n_pairs) put(__ldg(data + i), scale_of(i), i);
}

}  // namespace

int launch_dequant(const DequantArgs& a, const char** msg) {
  const int64_t elems = a.batch * a.rows * a.cols;
  if (elems == 0) return 0;
  const int64_t units = elems >> 3;  // 8 elements per thread step in every format
  int64_t blocks = (units + kThreads * kWordsPerLane - 1) / (kThreads * kWordsPerLane);
  const int64_t cap = static_cast<int64_t>(a.num_sms) * 8;
  if (blocks > cap) blocks = cap;
  const dim3 grid(static_cast<unsigned>(blocks)), block(kThreads);
  // FP8: the 16-byte form (one 16-byte load per lane per step, two steps in flight)
  if (a.fmt == BSQ_FP8_E4M3_B128 || a.fmt == BSQ_FP8_E4M3_TENSOR) {
    const int64_t loads = elems / 16;
    int64_t b16 = (loads + 2 * kThreads - 1) / (2 * kThreads);
    const int64_t cap16 = static_cast<int64_t>(a.num_sms) * 8;
    b16 = b16 < 1 ? 1 : (b16 > cap16 ? cap16 : b16);
    dequant_fp8_x2_kernel<<<dim3(static_cast<unsigned>(b16)), block, 0, a.stream>>>(
        static_cast<const uint4*>(a.data), static_cast<const float*>(a.scale), loads, a.rows, a.cols,
        fp8_scale_shift(a.fmt), static_cast<uint4*>(a.out));
    const cudaError_t e16 = cudaGetLastError();
    if (e16 != cudaSuccess) {
      *msg = cudaGetErrorString(e16);
      return static_cast<int>(e16);
    }
    return 0;
  }
  switch (a.fmt) {
    case BSQ_MXFP4:
      dequant_fp4_kernel<BSQ_MXFP4><<<grid, block, 0, a.stream>>>(
          static_cast<const uint32_t*>(a.data), static_cast<const uint8_t*>(a.scale), nullptr, units,
          a.rows * a.cols / 8, static_cast<uint4*>(a.out));
      break;
    case BSQ_NVFP4:
      dequant_fp4_kernel<BSQ_NVFP4><<<grid, block, 0, a.stream>>>(
          static_cast<const uint32_t*>(a.data), static_cast<const uint8_t*>(a.scale), a.tensor_scale, units,
          a.rows * a.cols / 8, static_cast<uint4*>(a.out));
      break;
    default:
      *msg = "bsq_dequant: format has no packed codes";
      return -1;
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *msg = cudaGetErrorString(e);
    return static_cast<int>(e);
  }
  return 0;
}

}  // namespace bsq
