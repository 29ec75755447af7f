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
//   FP8: blocks walk whole rows; consecutive lanes take consecutive 8-code units of a row
//        (8-byte loads, 16-byte stores, warp-contiguous), four rows in flight, and the
//        scale-block row is carried from row to row instead of divided out per unit.
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

// FP8 E4M3, row walk: block b takes the rows b, b + G, ... of the whole batch (G = grid
// size), four at a time; thread t takes the 8-code units t, t + 256, ... of each row, so a
// warp reads 256 and writes 512 contiguous bytes per instruction, four rows' loads in
// flight.  A row's batch entry and scale-block row are carried from step to step (a
// division only when a step passes more than one batch entry), one scale_inv per 8 codes.
__global__ void __launch_bounds__(kThreads) dequant_fp8_rows_kernel(const uint2* __restrict__ data,
                                                                    const float* __restrict__ scale_inv,
                                                                    int64_t total_rows, int64_t rows, int64_t cols,
                                                                    int shift, uint4* __restrict__ out) {
  const int64_t per_row = cols >> 3;
  const int64_t rblocks = shift >= 31 ? 1 : (rows + (1 << shift) - 1) >> shift;
  const int64_t cblocks = shift >= 31 ? 1 : (cols + (1 << shift) - 1) >> shift;
  const int64_t G = gridDim.x;
  // (batch entry, row inside it) of global row g, carried forward by `by` rows
  auto step = [&](int64_t& b, int64_t& r, int64_t by) {
    r += by;
    if (r >= rows) {
      if (r < 2 * rows) {   // the usual case: at most one batch entry passed
        r -= rows;
        ++b;
      } else {
        b += r / rows;
        r %= rows;
      }
    }
  };
  int64_t b0 = static_cast<int64_t>(blockIdx.x) / rows, r0 = static_cast<int64_t>(blockIdx.x) - b0 * rows;
  for (int64_t row = blockIdx.x; row < total_rows; row += 4 * G, step(b0, r0, 4 * G)) {
    int64_t bb[4], rr[4];
    bb[0] = b0;
    rr[0] = r0;
#pragma unroll
    for (int k = 1; k < 4; ++k) {
      bb[k] = bb[k - 1];
      rr[k] = rr[k - 1];
      step(bb[k], rr[k], G);
    }
    for (int64_t u = threadIdx.x; u < per_row; u += kThreads) {
      const int64_t cb = (u << 3) >> shift;
      uint2 w[4];
      float sv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t grow = row + k * G;
        w[k] = make_uint2(0u, 0u);
        sv[k] = 0.f;
        if (grow < total_rows) {
          w[k] = __ldg(data + grow * per_row + u);
          sv[k] = __ldg(scale_inv + (bb[k] * rblocks + (rr[k] >> shift)) * cblocks + cb);
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t grow = row + k * G;
        if (grow >= total_rows) continue;
        const ScaleBf16 s = make_scale_fp8(sv[k]);
        uint32_t a02, a13, b02, b13;
        decode_e4m3x4(w[k].x, s, a02, a13);
        decode_e4m3x4(w[k].y, s, b02, b13);
        uint4 o;
        unzip_pairs(a02, a13, o.x, o.y);  // (c0,c1), (c2,c3)
        unzip_pairs(b02, b13, o.z, o.w);  // (c4,c5), (c6,c7)
        out[grow * per_row + u] = o;
      }
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
  // FP8: the row walk, one block per row at a time (eight resident blocks per SM)
  if (a.fmt == BSQ_FP8_E4M3_B128 || a.fmt == BSQ_FP8_E4M3_TENSOR) {
    const int64_t trows = a.batch * a.rows;
    int64_t g = static_cast<int64_t>(a.num_sms) * 8;
    if (g > trows) g = trows;
    dequant_fp8_rows_kernel<<<dim3(static_cast<unsigned>(g)), block, 0, a.stream>>>(
        static_cast<const uint2*>(a.data), static_cast<const float*>(a.scale), trows, a.rows, a.cols,
        fp8_scale_shift(a.fmt), static_cast<uint4*>(a.out));
    const cudaError_t ef = cudaGetLastError();
    if (ef != cudaSuccess) {
      *msg = cudaGetErrorString(ef);
      return static_cast<int>(ef);
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
