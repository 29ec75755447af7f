// bsq_dequant.cu -- standalone dequantization of a packed operand to BF16 in HBM.
//
// The operation is the backward's "dequantize to BF16" step on its own
// (transformers PR #50031 `_dequantize_fp8_weight`; MSLK PR #393's FP4 dequantization
// helpers), used when a BF16 copy is wanted or as the first half of the
// dequantize-then-multiply path.  It is bound by HBM bandwidth: every warp reads
// contiguous 128-byte (FP4) / 256-byte (FP8) runs of packed codes and writes
// contiguous 512-byte runs of BF16 with 16-byte stores; scales are read once per
// 8 elements through the read-only path.
#include <cuda_bf16.h>

#include "bsq_decode.cuh"
#include "bsq_internal.h"
#include "../../include/bsq.h"

namespace bsq {

namespace {

constexpr int kThreads = 256;
constexpr int kWordsPerLane = 4;

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
        s = make_scale_nvfp4(sb[j], __ldg(tscale + idx / words_per_batch));
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

// FP8 E4M3 with square scale blocks of side 2^shift (128 x 128 blocks: shift 7; one scale
// per batch entry: shift 31): 8 codes (uint2) = 16 output bytes per unit.
__global__ void __launch_bounds__(kThreads) dequant_fp8_kernel(const uint2* __restrict__ data,
                                                               const float* __restrict__ scale_inv,
                                                               int64_t n_units, int64_t rows, int64_t cols,
                                                               int shift, uint4* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  const int64_t units_per_row = cols >> 3;
  const int64_t rblocks = shift >= 31 ? 1 : (rows + (1 << shift) - 1) >> shift;
  const int64_t cblocks = shift >= 31 ? 1 : (cols + (1 << shift) - 1) >> shift;
  constexpr int64_t kWarpUnits = 32 * kWordsPerLane;
  for (int64_t base = warp * kWarpUnits; base < n_units; base += nwarps * kWarpUnits) {
    uint2 w[kWordsPerLane];
    float sv[kWordsPerLane];
#pragma unroll
    for (int j = 0; j < kWordsPerLane; ++j) {
      const int64_t idx = base + lane + 32 * j;
      w[j] = make_uint2(0, 0);
      sv[j] = 0.f;
      if (idx < n_units) {
        w[j] = __ldg(data + idx);
        const int64_t grow = idx / units_per_row;          // row across the whole batch
        const int64_t col = (idx - grow * units_per_row) << 3;
        const int64_t b = grow / rows;
        const int64_t r = grow - b * rows;
        sv[j] = __ldg(scale_inv + (b * rblocks + (r >> shift)) * cblocks + (col >> shift));
      }
    }
#pragma unroll
    for (int j = 0; j < kWordsPerLane; ++j) {
      const int64_t idx = base + lane + 32 * j;
      if (idx >= n_units) continue;
      const ScaleBf16 s = make_scale_fp8(sv[j]);
      uint32_t a02, a13, b02, b13;
      decode_e4m3x4(w[j].x, s, a02, a13);
      decode_e4m3x4(w[j].y, s, b02, b13);
      uint4 o;
      unzip_pairs(a02, a13, o.x, o.y);  // (c0,c1), (c2,c3)
      unzip_pairs(b02, b13, o.z, o.w);  // (c4,c5), (c6,c7)
      out[idx] = o;
    }
  }
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
    case BSQ_FP8_E4M3_B128:
    case BSQ_FP8_E4M3_TENSOR:
      dequant_fp8_kernel<<<grid, block, 0, a.stream>>>(static_cast<const uint2*>(a.data),
                                                       static_cast<const float*>(a.scale), units, a.rows, a.cols,
                                                       fp8_scale_shift(a.fmt), static_cast<uint4*>(a.out));
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
