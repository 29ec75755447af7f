// bsq_decode.cuh -- register-level decode of packed E4M3 / E2M1 codes to BF16 with the
// block scale applied, bit-exact with the rule
//     out = RNE_bf16( bf16(code value) * RNE_bf16(scale) )
// (transformers PR #50031 `_dequantize_fp8_weight`: weight cast to the gradient dtype
// times the scale cast to that dtype; MSLK PR #393 "Implementation Method" for FP4).
//
// Technique.  A code's sign/exponent/mantissa bits are moved into the matching BF16
// bit positions without re-biasing the exponent.  The resulting BF16 number equals the
// code's value times a fixed power of two -- 2^-120 for E4M3 (bias 7 vs 127) and 2^-126
// for E2M1 (bias 1 vs 127) -- and this holds for subnormal codes too, because BF16 and
// the small formats share the same subnormal construction.  One BF16 multiply by the
// scale times the inverse power of two then yields RNE(value * scale) exactly, as long
// as that combined scale is itself a BF16 number ("fast" case); otherwise the value is
// first multiplied back exactly and then by the scale (two multiplies, same result).
//
// Two values whose code bits sit 16 bits apart in the packed word are built in one
// 32-bit operation, so the pairs produced are (c0,c4),(c1,c5),(c2,c6),(c3,c7) for FP4
// and (c0,c2),(c1,c3) for FP8 -- a fixed permutation inside every group of 8 elements
// that the consumers either undo (standalone dequant) or fold into their indexing
// (the GEMM maps tensor-memory lanes back to columns).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "../../include/bsq.h"

#include "bsq_ptx.cuh"

namespace bsq {

constexpr uint32_t kBf16NaN = 0x7FC0u;
constexpr uint32_t kPow2_126x2 = 0x7E807E80u;  // BF16 pair (2^126, 2^126)
constexpr uint32_t kPow2_120x2 = 0x7B807B80u;  // BF16 pair (2^120, 2^120)

// Position p of a decoded group of 8 holds element kPermFp4[p] (resp. kPermFp8[p]).
__host__ __device__ constexpr int perm_fp4(int p) { return (p & 1) ? (p >> 1) + 4 : (p >> 1); }
__host__ __device__ constexpr int perm_fp8(int p) {
  // (c0,c2),(c1,c3),(c4,c6),(c5,c7)
  return (p & 4) | ((p & 1) << 1) | ((p >> 1) & 1);
}

// A decoded 8-column group holds its columns in the order of the decode's BF16 pairs
// (perm_fp4 / perm_fp8 of the position); position i of a row of such groups holds column
// lane_to_col(i).
template <int FMT>
__device__ __forceinline__ int lane_to_col(int i) {
  if (FMT == BSQ_MXFP4 || FMT == BSQ_NVFP4) return (i & ~7) | perm_fp4(i & 7);
  if (FMT == BSQ_FP8_E4M3_B128) return (i & ~7) | perm_fp8(i & 7);
  return i;
}

struct ScaleBf16 {
  uint32_t s2;   // (s, s) BF16 pair
  uint32_t c2;   // (s * 2^k, s * 2^k) BF16 pair, valid when fast
  bool fast;
};

__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(f)));
}

// Combined scale for a code-to-BF16 offset of 2^-k (k = 126 for E2M1, 120 for E4M3).
__device__ __forceinline__ ScaleBf16 make_scale(uint32_t s_bits, float pow2k) {
  ScaleBf16 r;
  r.s2 = s_bits | (s_bits << 16);
  const float s = __uint_as_float(s_bits << 16);
  const float c = s * pow2k;  // exact in FP32 (a BF16 value shifted by a power of two) or +-inf
  // c is exactly a BF16 value (or inf/NaN): finite in BF16 iff |bits| <= BF16 max (0x7F7F0000).
  r.fast = (__float_as_uint(c) & 0x7FFFFFFFu) <= 0x7F7F0000u;
  const uint32_t cb = __float_as_uint(c) >> 16;
  r.c2 = cb | (cb << 16);
  return r;
}

// MXFP4: scale 2^(b-127); combined scale 2^(b-1) is a BF16 normal for b <= 128.
__device__ __forceinline__ ScaleBf16 make_scale_e8m0(uint32_t b) {
  ScaleBf16 r;
  const uint32_t s = (b == 255u) ? kBf16NaN : (b == 0u ? 0x0040u : (b << 7));
  r.s2 = s | (s << 16);
  r.fast = b <= 128u;
  const uint32_t c = (b + 126u) << 7;
  r.c2 = c | (c << 16);
  return r;
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  uint32_t h2;
  const uint16_t in = static_cast<uint16_t>(byte & 0xFFu);
  asm("{\n\t.reg .b16 t;\n\tmov.b16 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "h"(in));
  float f;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}

// NVFP4: scale = RNE_bf16( RNE_fp32(e4m3 block value * tensor scale) ).
__device__ __forceinline__ ScaleBf16 make_scale_nvfp4(uint32_t blk, float tensor_scale) {
  const float s = __fmul_rn(e4m3_to_f32(blk), tensor_scale);
  return make_scale(f32_to_bf16_bits(s), __uint_as_float(253u << 23) /* 2^126 */);
}

// FP8 blocks: scale = RNE_bf16(scale_inv).
__device__ __forceinline__ ScaleBf16 make_scale_fp8(float scale_inv) {
  return make_scale(f32_to_bf16_bits(scale_inv), __uint_as_float(247u << 23) /* 2^120 */);
}

__device__ __forceinline__ uint32_t apply_scale(uint32_t v2, const ScaleBf16& s, uint32_t pow2k_x2) {
  return s.fast ? bf16x2_mul(v2, s.c2) : bf16x2_mul(bf16x2_mul(v2, pow2k_x2), s.s2);
}

// Scaled-down BF16 pairs of 8 E2M1 codes (one 32-bit word, element j in bits 4j..4j+3):
// v[i] = (element i, element i+4), each = code value * 2^-126 with the code's sign.
// A nibble s|eem isolated at bit b is spread by one integer multiply into two copies,
// at b+6 (eem lands in BF16 exponent/mantissa bits 8:6) and b+12 (s lands in bit 15);
// the mask keeps those fields and drops the other halves of the copies.  The two
// nibbles of a pair sit 16 bits apart, so one multiply serves both.
__device__ __forceinline__ void spread_e2m1x8(uint32_t w, uint32_t (&v)[4]) {
  const uint32_t w8 = w >> 8;
  v[0] = ((w & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;   // nibbles at bits 0, 16: shifts 6 and 12
  v[1] = ((w & 0x00F000F0u) * 0x0104u) & 0x81C081C0u;   // nibbles at bits 4, 20: shifts 2 and 8
  v[2] = ((w8 & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;
  v[3] = ((w8 & 0x00F000F0u) * 0x0104u) & 0x81C081C0u;
}

__device__ __forceinline__ void scale_pairs4(uint32_t (&v)[4], const ScaleBf16& s, uint32_t pow2k_x2) {
  if (s.fast) {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = bf16x2_mul(v[i], s.c2);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = bf16x2_mul(bf16x2_mul(v[i], pow2k_x2), s.s2);
  }
}

// 8 E2M1 codes -> 4 BF16 pairs out[i] = (element i, element i+4), scaled.
__device__ __forceinline__ void decode_e2m1x8(uint32_t w, const ScaleBf16& s, uint32_t (&out)[4]) {
  spread_e2m1x8(w, out);
  scale_pairs4(out, s, kPow2_126x2);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Scaled-down BF16 pairs of 4 E4M3 codes (one word, element j in byte j):
// a = (c0, c2), b = (c1, c3), each = code value * 2^-120 (NaN codes not handled here).
// prmt puts each code in the low byte of its 16-bit half with a sign-filled byte above
// it; a 4-bit shift then lands the code's 7 magnitude bits (eeee.mmm) on BF16 bits 10..4
// and a sign copy on bit 15, and the mask clears the rest.
__device__ __forceinline__ void spread_e4m3x4(uint32_t w, uint32_t& a, uint32_t& b) {
  a = (prmt(w, 0u, 0xA280u) << 4) & 0x87F087F0u;
  b = (prmt(w, 0u, 0xB391u) << 4) & 0x87F087F0u;
}

// Bit 7 of byte j of the result is set exactly when byte j of w is an E4M3 NaN code
// (S.1111.111): the low seven bits plus one reach 0x80 only from 0x7F, and no carry leaves
// a byte.  Several words are tested at once by OR-ing their marks (not the words: an OR of
// codes gathers the bits of different codes and nearly always looks like 0x7F).
__device__ __forceinline__ uint32_t e4m3_nan_mark(uint32_t w) { return (w & 0x7F7F7F7Fu) + 0x01010101u; }
__device__ __forceinline__ bool e4m3_marked(uint32_t marks) { return (marks & 0x80808080u) != 0u; }
__device__ __forceinline__ bool e4m3_any_nan(uint32_t w) { return e4m3_marked(e4m3_nan_mark(w)); }

// Overwrite the NaN codes of word w in its decoded pairs with BF16 NaN.
__device__ __forceinline__ void e4m3_fix_nan(uint32_t w, uint32_t& p02, uint32_t& p13) {
  if ((w & 0x0000007Fu) == 0x0000007Fu) p02 = (p02 & 0xFFFF0000u) | kBf16NaN;
  if ((w & 0x00007F00u) == 0x00007F00u) p13 = (p13 & 0xFFFF0000u) | kBf16NaN;
  if ((w & 0x007F0000u) == 0x007F0000u) p02 = (p02 & 0x0000FFFFu) | (kBf16NaN << 16);
  if ((w & 0x7F000000u) == 0x7F000000u) p13 = (p13 & 0x0000FFFFu) | (kBf16NaN << 16);
}

// 4 E4M3 codes (one word, element j in byte j) -> 2 BF16 pairs (c0,c2),(c1,c3), scaled.
__device__ __forceinline__ void decode_e4m3x4(uint32_t w, const ScaleBf16& s, uint32_t& p02, uint32_t& p13) {
  spread_e4m3x4(w, p02, p13);
  p02 = apply_scale(p02, s, kPow2_120x2);
  p13 = apply_scale(p13, s, kPow2_120x2);
  // S.1111.111 is NaN in E4M3 (no infinities); the bit move above does not see it.
  if (e4m3_any_nan(w)) e4m3_fix_nan(w, p02, p13);
}

// 8 E4M3 codes (two words) -> one 8-element group as 4 BF16 pairs
// (c0,c2),(c1,c3),(c4,c6),(c5,c7), scaled.
__device__ __forceinline__ void decode_e4m3x8(uint32_t w0, uint32_t w1, const ScaleBf16& s, uint32_t (&out)[4]) {
  spread_e4m3x4(w0, out[0], out[1]);
  spread_e4m3x4(w1, out[2], out[3]);
  scale_pairs4(out, s, kPow2_120x2);
  if (e4m3_marked(e4m3_nan_mark(w0) | e4m3_nan_mark(w1))) {
    e4m3_fix_nan(w0, out[0], out[1]);
    e4m3_fix_nan(w1, out[2], out[3]);
  }
}

// 32 E4M3 codes of one row (lo = codes 0..15, hi = codes 16..31, element j of a word in
// byte j) -> groups out[g] = decode_e4m3x8 of codes 8g..8g+7, scaled; one exact NaN test
// covers all 32 codes, and only a row holding a NaN code takes the byte-by-byte fix.
__device__ __forceinline__ void decode_e4m3x32(const uint4& lo, const uint4& hi, const ScaleBf16& s,
                                               uint32_t (&out)[4][4]) {
  spread_e4m3x4(lo.x, out[0][0], out[0][1]);
  spread_e4m3x4(lo.y, out[0][2], out[0][3]);
  spread_e4m3x4(lo.z, out[1][0], out[1][1]);
  spread_e4m3x4(lo.w, out[1][2], out[1][3]);
  spread_e4m3x4(hi.x, out[2][0], out[2][1]);
  spread_e4m3x4(hi.y, out[2][2], out[2][3]);
  spread_e4m3x4(hi.z, out[3][0], out[3][1]);
  spread_e4m3x4(hi.w, out[3][2], out[3][3]);
#pragma unroll
  for (int g = 0; g < 4; ++g) scale_pairs4(out[g], s, kPow2_120x2);
  if (e4m3_marked(e4m3_nan_mark(lo.x) | e4m3_nan_mark(lo.y) | e4m3_nan_mark(lo.z) | e4m3_nan_mark(lo.w) |
                  e4m3_nan_mark(hi.x) | e4m3_nan_mark(hi.y) | e4m3_nan_mark(hi.z) | e4m3_nan_mark(hi.w))) {
    e4m3_fix_nan(lo.x, out[0][0], out[0][1]);
    e4m3_fix_nan(lo.y, out[0][2], out[0][3]);
    e4m3_fix_nan(lo.z, out[1][0], out[1][1]);
    e4m3_fix_nan(lo.w, out[1][2], out[1][3]);
    e4m3_fix_nan(hi.x, out[2][0], out[2][1]);
    e4m3_fix_nan(hi.y, out[2][2], out[2][3]);
    e4m3_fix_nan(hi.z, out[3][0], out[3][1]);
    e4m3_fix_nan(hi.w, out[3][2], out[3][3]);
  }
}

// Undo the pair permutation: pairs (x_lo, x_hi),(y_lo, y_hi) -> (x_lo, y_lo),(x_hi, y_hi).
__device__ __forceinline__ void unzip_pairs(uint32_t x, uint32_t y, uint32_t& lo, uint32_t& hi) {
  lo = prmt(x, y, 0x5410u);
  hi = prmt(x, y, 0x7632u);
}

}  // namespace bsq
