// bsq_smallm.cu -- dgrad for a handful of token rows (M <= 16): grad_X[M,K] = grad_out[M,N] @ deq(W)[N,K]
// (MSLK PR #393 "Implementation Method"; transformers PR #50031 `FP8LinearFunction.backward`).
//
// With M this small the product is bound by reading the packed weight once from HBM, so
// the kernel is shaped for bandwidth, not for the tensor-core peak:
//   * split-K over the N rows of W: every CTA owns a 128-column slab of K and a range of
//     up to 512 rows, so that about two CTAs per SM cover W in one wave;
//   * one thread stages the CTA's whole W slab, its scale slab and the matching grad_out
//     slab into shared memory with TMA behind a single barrier, so all of W is in flight
//     at once and the kernel runs at memory speed rather than at memory latency;
//   * decoding pairs the same column of two adjacent rows in one 32-bit register
//     (one byte permute + the multiply-spread of bsq_decode.cuh), which is exactly the
//     k-pair an mma.sync B fragment wants, so no transpose and no BF16 staging is needed;
//   * m16n8k16 BF16 mma.sync with FP32 accumulators (tokens are the M=16 side);
//   * the warps of a CTA reduce through shared memory.  The row splits of a slab then add
//     up in one of two ways: smallm_dgrad_cluster_kernel (bsq_linear_dgrad) makes them one
//     thread-block cluster and adds through distributed shared memory; smallm_dgrad_kernel
//     (the allocation-free entry point) adds into an FP32 scratch with 16-byte reduction
//     atomics, and the last CTA of a slab converts it to BF16, writes grad_X and zeroes the
//     scratch again.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "bsq_decode.cuh"
#include "bsq_internal.h"
#include "bsq_ptx.cuh"
#include "../../include/bsq.h"

namespace bsq {

bool encode_map(CUtensorMap* m, CUtensorMapDataType dt, uint32_t rank, const void* base, const uint64_t* dims,
                const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle sw);

namespace {

constexpr int kWarps = 8;
constexpr int kThreadsSm = kWarps * 32;
constexpr int kSlab = 128;       // columns of K per CTA
constexpr int kStep = 16;        // rows of N per mma k-step
constexpr int kNT = 16;          // n-tiles (8 columns each) per warp per k-step
constexpr int kMaxRows = 512;    // rows of W per CTA
constexpr int kBox = 256;        // rows per TMA box

struct SmallParams {
  const uint8_t* scale;
  const float* tensor_scale;
  __nv_bfloat16* out;
  float* ws;          // [16][K] FP32, all zero between calls
  int32_t* counters;  // [num_slabs], all zero between calls
  int32_t M, N, K;
  int32_t rows_per_split;   // multiple of kStep * kWarps, <= kMaxRows
  int32_t scale_ld;         // MXFP4: K/32, NVFP4: K/16, FP8: ceil(K/128)
  int32_t scale_tma;        // FP4 scale slab through TMA
  uint64_t timeout_ns;
  int32_t* err;
};

template <int FMT>
struct SmallFmt {
  static constexpr int kRowBytes = FMT == BSQ_FP8_E4M3_B128 ? kSlab : kSlab / 2;
  static constexpr int kWBytes = kMaxRows * kRowBytes;
  static constexpr int kSBytes = FMT == BSQ_FP8_E4M3_B128 ? 0 : kMaxRows * 16;
  static constexpr int kGBytes = 16 * kMaxRows * 2;
  static constexpr int kRedBytes = kWarps * kNT * 16 * 8 * 4;   // per-warp partial slabs
  static constexpr int kStageBytes = kWBytes + kSBytes + kGBytes;
  // staged slabs (later reused for the partials), the summed slab, the barrier and the flag;
  // plus 1 KB to align the base for the 128-byte swizzled grad_out boxes
  static constexpr int kSmem = (kStageBytes > kRedBytes ? kStageBytes : kRedBytes) + 16 * kSlab * 4 + 128 + 1024;
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
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
__device__ __forceinline__ ScaleBf16 row_scale(uint32_t raw, float tscale) {
  if (FMT == BSQ_MXFP4) return make_scale_e8m0(raw);
  return make_scale_nvfp4(raw, tscale);
}

template <int FMT>
__global__ void __launch_bounds__(kThreadsSm, 2)
    smallm_dgrad_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s,
                        const __grid_constant__ CUtensorMap tm_g, const SmallParams p) {
  using F = SmallFmt<FMT>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kStaged = F::kStageBytes > F::kRedBytes ? F::kStageBytes : F::kRedBytes;
  uint8_t* ws_w = base;                               // [rows][kRowBytes] packed W
  uint8_t* ws_s = ws_w + F::kWBytes;                  // [rows][16] FP4 scale windows
  uint8_t* ws_g = ws_s + F::kSBytes;                  // [rows/64][16 tokens][64] BF16 grad_out, 128B-swizzled
  float* red = reinterpret_cast<float*>(base);        // reused after the main loop
  float* red_sum = reinterpret_cast<float*>(base + kStaged);
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + kStaged + 16 * kSlab * 4);
  int* last_flag = reinterpret_cast<int*>(base + kStaged + 16 * kSlab * 4 + 64);
  const int slab = blockIdx.x;
  const int cb = slab * kSlab;
  const int n0 = blockIdx.y * p.rows_per_split;
  const int n1 = min(p.N, n0 + p.rows_per_split);
  const int nrows = max(n1 - n0, 0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;

  if (tid == 0) {
    mbar_init(smem_u32(bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    const int nbox = (nrows + kBox - 1) / kBox;
    const int ngbox = (nrows + 63) / 64;
    uint32_t bytes = nbox * kBox * F::kRowBytes + ngbox * 16 * 64 * 2;
    if (F::kSBytes && p.scale_tma) bytes += nbox * kBox * 16;
    mbar_arrive_expect_tx(smem_u32(bar), bytes);
    for (int b = 0; b < nbox; ++b) {
      const int row = n0 + b * kBox;
      tma_load_2d(smem_u32(ws_w + b * kBox * F::kRowBytes), &tm_w, smem_u32(bar),
                  FMT == BSQ_FP8_E4M3_B128 ? cb : cb / 2, row);
      if (F::kSBytes && p.scale_tma)
        tma_load_2d(smem_u32(ws_s + b * kBox * 16), &tm_s, smem_u32(bar),
                    (FMT == BSQ_MXFP4 ? (cb >> 5) : (cb >> 4)) & ~15, row);
    }
    for (int b = 0; b < ngbox; ++b)   // [16 tokens][64 rows] per box, 16-byte chunks XOR-swizzled by token
      tma_load_2d(smem_u32(ws_g + b * 16 * 64 * 2), &tm_g, smem_u32(bar), n0 + 64 * b, 0);
  }
  float tscale = 0.f;
  if (FMT == BSQ_NVFP4) tscale = __ldg(p.tensor_scale);
  const int col = cb + 16 * g;
  const bool col_ok = col < p.K;
  float acc[kNT][4];
#pragma unroll
  for (int i = 0; i < kNT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  // bounded wait for the slab; the CTA takes one decision (a thread that gave up stops all)
  bool ok = true;
  {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait_sleep(smem_u32(bar), 0, 20000u)) {
      if (global_timer_ns() - t0 > p.timeout_ns) {
        ok = false;
        break;
      }
    }
  }
  ok = __syncthreads_and(ok) != 0;
  if (ok) {
    const int nsteps = (nrows + kStep - 1) / kStep;
    for (int ks = warp; ks < nsteps; ks += kWarps) {
      const int lr = ks * kStep;               // local row of this k-step
      const int rows[4] = {lr + 2 * q, lr + 2 * q + 1, lr + 8 + 2 * q, lr + 9 + 2 * q};
      // A fragment: grad_out[token][k] for k = local rows lr .. lr+15, read from the swizzled
      // boxes ([16 tokens][64 rows], chunk of 8 rows XOR token & 7): conflict-free
      const uint32_t gb = smem_u32(ws_g + (lr >> 6) * 16 * 64 * 2);
      const int kl = lr & 63;                     // multiple of 16: chunks kl/8 and kl/8 + 1
      const uint32_t c0 = static_cast<uint32_t>(((kl >> 3) ^ (g & 7)) << 4);
      const uint32_t c1 = static_cast<uint32_t>((((kl >> 3) + 1) ^ (g & 7)) << 4);
      uint32_t a[4];
      a[0] = lds_u32(gb + g * 128 + c0 + 4 * q);
      a[1] = lds_u32(gb + (g + 8) * 128 + c0 + 4 * q);
      a[2] = lds_u32(gb + g * 128 + c1 + 4 * q);
      a[3] = lds_u32(gb + (g + 8) * 128 + c1 + 4 * q);
      if (FMT == BSQ_FP8_E4M3_B128) {
        float sf = 0.f;
        if (col_ok && n0 + lr < n1)
          sf = __ldg(reinterpret_cast<const float*>(p.scale) + static_cast<int64_t>((n0 + lr) >> 7) * p.scale_ld + (col >> 7));
        const ScaleBf16 sc = make_scale_fp8(sf);
        uint4 w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = *reinterpret_cast<const uint4*>(ws_w + rows[i] * F::kRowBytes + 16 * g);
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
          uint32_t b0[4], b1[4];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint32_t* xw = reinterpret_cast<const uint32_t*>(&w[2 * half]);
            const uint32_t* yw = reinterpret_cast<const uint32_t*>(&w[2 * half + 1]);
            uint32_t(&dst)[4] = half ? b1 : b0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t v = pair_bytes(xw[wi], yw[wi], j);   // column 4wi+j of both rows
              uint32_t o = scale_one(((v << 4) & 0x07F007F0u) | ((v << 8) & 0x80008000u), sc, kPow2_120x2);
              if ((v & 0x7Fu) == 0x7Fu) o = (o & 0xFFFF0000u) | kBf16NaN;                 // E4M3 NaN, first row
              if ((v & 0x007F0000u) == 0x007F0000u) o = (o & 0xFFFFu) | (kBf16NaN << 16);  // second row
              dst[j] = o;
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) mma_bf16_16816(acc[4 * wi + j], a, b0[j], b1[j]);
        }
      } else {
        uint2 w[4];
        uint32_t sraw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          w[i] = *reinterpret_cast<const uint2*>(ws_w + rows[i] * F::kRowBytes + 8 * g);
          const int grow = n0 + rows[i];
          if (p.scale_tma) {
            sraw[i] = FMT == BSQ_MXFP4 ? ws_s[rows[i] * 16 + ((cb >> 5) & 15) + (g >> 1)]
                                       : ws_s[rows[i] * 16 + ((cb >> 4) & 15) + g];
          } else {
            sraw[i] = 0;
            if (col_ok && grow < n1)
              sraw[i] = __ldg(p.scale + static_cast<int64_t>(grow) * p.scale_ld + (FMT == BSQ_MXFP4 ? (col >> 5) : (col >> 4)));
          }
        }
#pragma unroll
        for (int wi = 0; wi < 2; ++wi) {
          uint32_t b0[8], b1[8];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint32_t* xw = reinterpret_cast<const uint32_t*>(&w[2 * half]);
            const uint32_t* yw = reinterpret_cast<const uint32_t*>(&w[2 * half + 1]);
            const ScaleBf16 sc = pair_scales(row_scale<FMT>(sraw[2 * half], tscale), row_scale<FMT>(sraw[2 * half + 1], tscale));
            uint32_t(&dst)[8] = half ? b1 : b0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t v = pair_bytes(xw[wi], yw[wi], j);                   // byte 4wi+j of both rows
              dst[2 * j] = scale_one(((v & 0x000F000Fu) * 0x1040u) & 0x81C081C0u, sc, kPow2_126x2);     // column 8wi+2j
              dst[2 * j + 1] = scale_one(((v & 0x00F000F0u) * 0x0104u) & 0x81C081C0u, sc, kPow2_126x2);  // 8wi+2j+1
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) mma_bf16_16816(acc[8 * wi + j], a, b0[j], b1[j]);
        }
      }
    }
  }
  if (!ok) {
    // Orderly abort: record the timeout, give the copies still in flight one more bounded
    // wait to land (nothing reads or reuses the staged region), write nothing, and keep
    // only the workspace bookkeeping: the last CTA of the slab re-zeroes the slab's
    // workspace and counter so later calls start clean.  grad_X of this call is undefined.
    if (tid == 0) {
      atomicCAS(p.err, 0, BSQ_DEVERR_TIMEOUT);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(smem_u32(bar), 0) && global_timer_ns() - t0 < kDrainLimitNs) {
      }
    }
    __syncthreads();
    if (gridDim.y == 1) return;
    __threadfence();
    if (tid == 0) *last_flag = (atomicAdd(p.counters + slab, 1) == static_cast<int>(gridDim.y) - 1);
    __syncthreads();
    if (!*last_flag) return;
    __threadfence();
    for (int i = tid; i < 16 * kSlab / 4; i += kThreadsSm) {
      const int t = (4 * i) / kSlab, c = cb + (4 * i) % kSlab;
      if (t < p.M && c < p.K) __stcg(reinterpret_cast<float4*>(p.ws + static_cast<int64_t>(t) * p.K + c),
                                     make_float4(0.f, 0.f, 0.f, 0.f));
    }
    if (tid == 0) p.counters[slab] = 0;
    return;
  }
  __syncthreads();   // everyone is done with the staged slabs; reuse them for the partials

  // Per-warp partial slabs laid out [nt][token][n] (8-byte stores of fragment column pairs);
  // fragment column n of n-tile nt is output column cb + 16 n + nt.
  {
    float* mine = red + warp * (kNT * 16 * 8);
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      *reinterpret_cast<float2*>(mine + (nt * 16 + g) * 8 + 2 * q) = make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2*>(mine + (nt * 16 + g + 8) * 8 + 2 * q) = make_float2(acc[nt][2], acc[nt][3]);
    }
  }
  __syncthreads();
  // Sum the warps into red_sum laid out [token][128 columns]; entries are read in their
  // own order (conflict-free) and scattered: entry (nt, token t, n) -> column 16 n + nt.
  for (int e = tid; e < 16 * kSlab; e += kThreadsSm) {
    const int n = e & 7, t = (e >> 3) & 15, nt = e >> 7;
    float v = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) v += red[w2 * (kNT * 16 * 8) + e];
    red_sum[t * kSlab + 16 * n + nt] = v;
  }
  __syncthreads();

  if (gridDim.y == 1) {
    for (int i = tid; i < 16 * kSlab; i += kThreadsSm) {
      const int t = i / kSlab, c = cb + i % kSlab;
      if (t < p.M && c < p.K) p.out[static_cast<int64_t>(t) * p.K + c] = __float2bfloat16_rn(red_sum[i]);
    }
    return;
  }
  // 16-byte reduction atomics into the workspace (K % 16 == 0 keeps them aligned)
  for (int i = tid; i < 16 * kSlab / 4; i += kThreadsSm) {
    const int t = (4 * i) / kSlab, c = cb + (4 * i) % kSlab;
    if (t < p.M && c < p.K)
      red_add_v4(p.ws + static_cast<int64_t>(t) * p.K + c, red_sum[4 * i], red_sum[4 * i + 1], red_sum[4 * i + 2],
                 red_sum[4 * i + 3]);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) *last_flag = (atomicAdd(p.counters + slab, 1) == static_cast<int>(gridDim.y) - 1);
  __syncthreads();
  if (!*last_flag) return;
  __threadfence();
  for (int i = tid; i < 16 * kSlab / 4; i += kThreadsSm) {
    const int t = (4 * i) / kSlab, c = cb + (4 * i) % kSlab;
    if (t < p.M && c < p.K) {
      float4* w = reinterpret_cast<float4*>(p.ws + static_cast<int64_t>(t) * p.K + c);
      const float4 v = __ldcg(w);
      __stcg(w, make_float4(0.f, 0.f, 0.f, 0.f));
      __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(p.out + static_cast<int64_t>(t) * p.K + c) = pk;
    }
  }
  if (tid == 0) p.counters[slab] = 0;
}

// ---------------------------------------------------------------- cluster-reduced variant
// The same product without any global workspace, for one weight (bsq_linear_dgrad) or for
// the experts of a grouped dgrad (bsq_grouped_dgrad): the CTAs that split a column slab's
// rows form one thread-block cluster and add their partial sums through distributed
// shared memory.  Each CTA streams its rows in 64-row chunks, each chunk on its own
// barrier, so decoding starts with the first chunk instead of after the whole slab.
//
// Grouped, every CTA builds the same list of experts that have rows for this kernel from
// the device offsets (validated first; nothing is written when they are malformed), and
// walks the list with stride gridDim.z.  An expert's rows go through in passes of up to
// 16 tokens; every pass streams the expert's W slab again (from L2 after the first).
constexpr int kChunk = 64;        // rows of W per TMA chunk (four mma k-steps)
constexpr int kRing = 8;          // chunks in flight per CTA
constexpr int kMaxSplits = 8;     // CTAs of a cluster (portable cluster size)
constexpr int kTok = 16;          // token rows per pass (the mma M side)
constexpr int kScaleStage = 128;  // FP8 scale blocks of a CTA's rows staged in shared memory
static_assert(kMaxExperts <= 4 * kThreadsSm, "the expert scan gives each thread four experts");

struct ClusterParams {
  const uint8_t* scale;
  const float* tensor_scale;  // NVFP4: one per expert
  __nv_bfloat16* out;         // bf16 [S][K]
  const int32_t* offsets;     // cumulative end offsets [E]; null: one group of S rows
  int64_t scale_batch;        // scale entries per expert (FP8: floats; FP4: bytes)
  int32_t S, N, K, E;
  int32_t rows_per_split;     // multiple of kChunk
  int32_t scale_ld;           // MXFP4: K/32, NVFP4: K/16, FP8: ceil(K/128) (1 with one scale per tensor)
  int32_t scale_shift;        // FP8: log2 of the scale block's side (7; 31 for one scale per tensor)
  int32_t scale_tma;          // FP4 scale windows through TMA
  int32_t tail_rows;          // grouped: an expert's last (rows % kTileN) rows are this kernel's when 1..tail_rows
  int32_t drop_chunk;         // test hook: every CTA's first chunk is never copied (its wait runs out)
  uint64_t timeout_ns;
  int32_t* err;
};

template <int FMT>
struct ClusterFmt {
  static constexpr int kRowBytes = FMT == BSQ_FP8_E4M3_B128 ? kSlab : kSlab / 2;
  static constexpr int kWBytes = kChunk * kRowBytes;
  static constexpr int kSBytes = FMT == BSQ_FP8_E4M3_B128 ? 0 : kChunk * 16;
  static constexpr int kGBytes = kTok * kChunk * 2;   // [16 tokens][64 rows] BF16, 128-byte swizzled
  static constexpr int kSlotBytes = kWBytes + kSBytes + kGBytes;
  static_assert(kSlotBytes % 1024 == 0, "swizzled grad_out boxes need 1024-byte aligned slots");
  static constexpr int kRingBytes = kRing * kSlotBytes;
  static constexpr int kTreeBytes = kWarps * kTok * kSlab * 4;   // partials of the eight warps
  static constexpr int kStaged = kRingBytes > kTreeBytes ? kRingBytes : kTreeBytes;
  static constexpr int kRedBytes = kTok * kSlab * 4;      // this CTA's partial, read by the cluster
  static constexpr int kBarBytes = 256;                   // barriers, counters, status words
  static constexpr int kScaleBytes = kScaleStage * 4;     // FP8: the pass's scales of this slab
  static constexpr int kListBytes = kMaxExperts * 2;      // experts with rows for this kernel
  static constexpr int kSmem = kStaged + kRedBytes + kBarBytes + kScaleBytes + kListBytes + 1024;
};

// The rows [t0, t1) of expert e that this kernel computes.
__device__ __forceinline__ void expert_rows(const ClusterParams& p, int e, int& t0, int& t1) {
  if (!p.offsets) {
    t0 = 0;
    t1 = p.S;
    return;
  }
  const int r0 = e ? __ldg(p.offsets + e - 1) : 0, r1 = __ldg(p.offsets + e);
  const int tail = (r1 - r0) % kTileN;
  t1 = r1;
  t0 = (tail > 0 && tail <= p.tail_rows) ? r1 - tail : r1;
}

template <int FMT>
__global__ void __launch_bounds__(kThreadsSm, 2)
    smallm_dgrad_cluster_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s,
                                const __grid_constant__ CUtensorMap tm_g, const ClusterParams p) {
  using F = ClusterFmt<FMT>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* tree = reinterpret_cast<float*>(base);                  // warp partials; reuse the ring after a pass
  float* red = reinterpret_cast<float*>(base + F::kStaged);      // [16 tokens][128 columns]
  uint64_t* full = reinterpret_cast<uint64_t*>(base + F::kStaged + F::kRedBytes);
  uint32_t* released = reinterpret_cast<uint32_t*>(full + kRing);   // per slot: warps done with it, ever
  int32_t* fills = reinterpret_cast<int32_t*>(released + kRing);     // copies issued into each slot
  int32_t* pass_ok = fills + kRing;                              // this CTA's pass went through (read by the cluster)
  int32_t* n_items = pass_ok + 1;
  int32_t* warp_sum = n_items + 1;                               // [kWarps] scan of the expert list
  float* scale_s = reinterpret_cast<float*>(base + F::kStaged + F::kRedBytes + F::kBarBytes);
  int16_t* items = reinterpret_cast<int16_t*>(base + F::kStaged + F::kRedBytes + F::kBarBytes + F::kScaleBytes);
  const int slab = blockIdx.x;
  const int cb = slab * kSlab;
  const int n0 = blockIdx.y * p.rows_per_split;
  const int n1 = min(p.N, n0 + p.rows_per_split);
  const int nchunks = n1 > n0 ? (n1 - n0 + kChunk - 1) / kChunk : 0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const int grp = warp >> 2;         // warps 0-3 take even chunks, 4-7 odd ones
  const int kstep = warp & 3;        // the warp's 16-row k-step of a chunk
  const uint32_t crank = cluster_ctarank();
  const uint32_t csize = gridDim.y;  // the cluster spans the row splits of one slab

  if (tid == 0) {
    for (int s = 0; s < kRing; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      released[s] = 0;
      fills[s] = 0;
    }
    fence_mbar_init();
  }
  // The experts with rows here, in increasing order (the same list in every CTA).
  if (p.offsets) {
    int bad = 0, cnt = 0;
    uint32_t has = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = 4 * tid + j;
      if (e < p.E) {
        const int r0 = e ? __ldg(p.offsets + e - 1) : 0, r1 = __ldg(p.offsets + e);
        if (r1 < r0 || r1 > p.S || r0 < 0) bad = 1;
        const int tail = (r1 - r0) % kTileN;
        if (tail > 0 && tail <= p.tail_rows) {
          has |= 1u << j;
          ++cnt;
        }
      }
    }
    if (__syncthreads_or(bad)) {
      // every CTA of the grid reads the same offsets and leaves here, before any copy
      if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
        atomicCAS(p.err, 0, BSQ_DEVERR_BAD_OFFSETS);
      return;
    }
    int incl = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    int pos = incl - cnt;
    for (int w2 = 0; w2 < warp; ++w2) pos += warp_sum[w2];
    if (tid == kThreadsSm - 1) *n_items = pos + cnt;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if ((has >> j) & 1u) items[pos++] = static_cast<int16_t>(4 * tid + j);
  } else if (tid == 0) {
    *n_items = 1;
    items[0] = 0;
  }
  __syncthreads();
  const int num_items = *n_items;

  auto slot_of = [&](uint32_t cc) { return base + (cc % kRing) * F::kSlotBytes; };
  // TMA of the pass's chunk c (ring position cc) of expert e, token rows from r0
  auto issue = [&](uint32_t cc, int c, int e, int r0) {
    if (p.drop_chunk && cc == 0) return;
    uint8_t* s = slot_of(cc);
    fills[cc % kRing] += 1;
    const uint32_t bar = smem_u32(&full[cc % kRing]);
    const int row = n0 + c * kChunk;
    mbar_arrive_expect_tx(bar, F::kWBytes + ((F::kSBytes && p.scale_tma) ? F::kSBytes : 0) + F::kGBytes);
    tma_load_3d(smem_u32(s), &tm_w, bar, FMT == BSQ_FP8_E4M3_B128 ? cb : cb / 2, row, e);
    if (F::kSBytes && p.scale_tma)
      tma_load_3d(smem_u32(s + F::kWBytes), &tm_s, bar, (FMT == BSQ_MXFP4 ? (cb >> 5) : (cb >> 4)) & ~15, row, e);
    tma_load_2d(smem_u32(s + F::kWBytes + F::kSBytes), &tm_g, bar, row, r0);
  };

  const int col = cb + 16 * g;
  const bool col_ok = col < p.K;
  uint32_t cbase = 0;    // ring position of the pass's first chunk
  bool live = true;      // every pass so far went through in every CTA of the cluster
  for (int it = blockIdx.z; it < num_items && live; it += gridDim.z) {
    const int e = items[it];
    int t0, t1;
    expert_rows(p, e, t0, t1);
    float tscale = 0.f;
    if (FMT == BSQ_NVFP4) tscale = __ldg(p.tensor_scale + e);
    const uint8_t* scale_e = p.scale + p.scale_batch * e * (FMT == BSQ_FP8_E4M3_B128 ? 4 : 1);
    // FP8: this slab's scales of the CTA's rows, one per scale block (one per tensor: one)
    const int sb0 = n0 >> p.scale_shift;
    const int nsb = n1 > n0 ? ((n1 - 1) >> p.scale_shift) - sb0 + 1 : 0;
    const bool staged = FMT == BSQ_FP8_E4M3_B128 && nsb <= kScaleStage;
    if (staged) {
      const float* sc = reinterpret_cast<const float*>(scale_e);
      for (int i = tid; i < nsb; i += kThreadsSm)
        scale_s[i] = __ldg(sc + static_cast<int64_t>(sb0 + i) * p.scale_ld + (cb >> p.scale_shift));
      __syncthreads();
    }
    for (int r0 = t0; r0 < t1 && live; r0 += kTok) {
      const int mt = min(kTok, t1 - r0);
      if (tid == 0)
        for (int c = 0; c < min(nchunks, kRing); ++c) issue(cbase + c, c, e, r0);
      float acc[kNT][4];
#pragma unroll
      for (int i = 0; i < kNT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

      bool ok = true;
      for (int c = grp; c < nchunks; c += 2) {
        const uint32_t cc = cbase + c;
        const uint32_t si = cc % kRing;
        const uint32_t par = (cc / kRing) & 1u;
        if (!mbar_try_wait(smem_u32(&full[si]), par)) {
          const uint64_t w0 = global_timer_ns();
          while (!mbar_try_wait_sleep(smem_u32(&full[si]), par, 20000u)) {
            if (global_timer_ns() - w0 > p.timeout_ns) {
              ok = false;
              break;
            }
          }
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const uint8_t* ws_w = slot_of(cc);
        const uint8_t* ws_s = ws_w + F::kWBytes;
        const uint32_t gb = smem_u32(ws_w + F::kWBytes + F::kSBytes);
        const int lr = kstep * kStep;                 // the k-step's first row inside the chunk
        const int grow0 = n0 + c * kChunk + lr;       // its row of W
        // A fragment: grad_out[token][k], k = the k-step's 16 rows (chunk lr/8, lr/8 + 1 of the
        // 128-byte swizzled [16 tokens][64 rows] box)
        const uint32_t c0 = static_cast<uint32_t>(((lr >> 3) ^ (g & 7)) << 4);
        const uint32_t c1 = static_cast<uint32_t>((((lr >> 3) + 1) ^ (g & 7)) << 4);
        uint32_t a[4];
        a[0] = lds_u32(gb + g * 128 + c0 + 4 * q);
        a[1] = lds_u32(gb + (g + 8) * 128 + c0 + 4 * q);
        a[2] = lds_u32(gb + g * 128 + c1 + 4 * q);
        a[3] = lds_u32(gb + (g + 8) * 128 + c1 + 4 * q);
        if (FMT == BSQ_FP8_E4M3_B128) {
          float sf;
          if (staged) {
            sf = scale_s[min((grow0 >> p.scale_shift) - sb0, nsb - 1)];
          } else {
            sf = 0.f;
            if (col_ok && grow0 < n1)
              sf = __ldg(reinterpret_cast<const float*>(scale_e) + static_cast<int64_t>(grow0 >> p.scale_shift) * p.scale_ld +
                         (col >> p.scale_shift));
          }
          const ScaleBf16 sc = make_scale_fp8(sf);   // one scale block holds the whole k-step
          // rows lr+2q, lr+2q+1, lr+8+2q, lr+9+2q, 16 codes each from column 16g: 16-byte
          // chunk g of a 128-byte row, stored at chunk g ^ (row & 7) (128-byte swizzle)
          uint4 w[4];
          const uint32_t wrow = smem_u32(ws_w) + static_cast<uint32_t>(lr + 2 * q) * F::kRowBytes;
          w[0] = lds128(wrow + ((g ^ (2 * q)) << 4));
          w[1] = lds128(wrow + F::kRowBytes + ((g ^ (2 * q + 1)) << 4));
          w[2] = lds128(wrow + 8 * F::kRowBytes + ((g ^ (2 * q)) << 4));
          w[3] = lds128(wrow + 9 * F::kRowBytes + ((g ^ (2 * q + 1)) << 4));
          const bool any_nan = e4m3_marked(
              e4m3_nan_mark(w[0].x) | e4m3_nan_mark(w[0].y) | e4m3_nan_mark(w[0].z) | e4m3_nan_mark(w[0].w) |
              e4m3_nan_mark(w[1].x) | e4m3_nan_mark(w[1].y) | e4m3_nan_mark(w[1].z) | e4m3_nan_mark(w[1].w) |
              e4m3_nan_mark(w[2].x) | e4m3_nan_mark(w[2].y) | e4m3_nan_mark(w[2].z) | e4m3_nan_mark(w[2].w) |
              e4m3_nan_mark(w[3].x) | e4m3_nan_mark(w[3].y) | e4m3_nan_mark(w[3].z) | e4m3_nan_mark(w[3].w));
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            uint32_t b0[4], b1[4];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const uint32_t* xw = reinterpret_cast<const uint32_t*>(&w[2 * half]);
              const uint32_t* yw = reinterpret_cast<const uint32_t*>(&w[2 * half + 1]);
              uint32_t(&dst)[4] = half ? b1 : b0;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                // byte j of both rows, each in the low byte of its 16-bit half with a sign-filled
                // byte above it; a 4-bit shift puts the magnitude bits on BF16 bits 10..4 and the
                // sign on bit 15 (code value x 2^-120)
                const uint32_t v = prmt(xw[wi], yw[wi], static_cast<uint32_t>(j | ((j | 8) << 4) | ((4 + j) << 8) |
                                                                                  (((4 + j) | 8) << 12)));
                dst[j] = (v << 4) & 0x87F087F0u;
              }
            }
            if (sc.fast) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                b0[j] = bf16x2_mul(b0[j], sc.c2);
                b1[j] = bf16x2_mul(b1[j], sc.c2);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                b0[j] = bf16x2_mul(bf16x2_mul(b0[j], kPow2_120x2), sc.s2);
                b1[j] = bf16x2_mul(bf16x2_mul(b1[j], kPow2_120x2), sc.s2);
              }
            }
            if (any_nan) {
              // S.1111.111 is NaN in E4M3; the bit move above does not see it
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                const uint32_t* xw = reinterpret_cast<const uint32_t*>(&w[2 * half]);
                const uint32_t* yw = reinterpret_cast<const uint32_t*>(&w[2 * half + 1]);
                uint32_t(&dst)[4] = half ? b1 : b0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  if (((xw[wi] >> (8 * j)) & 0x7Fu) == 0x7Fu) dst[j] = (dst[j] & 0xFFFF0000u) | kBf16NaN;
                  if (((yw[wi] >> (8 * j)) & 0x7Fu) == 0x7Fu) dst[j] = (dst[j] & 0xFFFFu) | (kBf16NaN << 16);
                }
              }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) mma_bf16_16816(acc[4 * wi + j], a, b0[j], b1[j]);
          }
        } else {
          // rows lr+2q, lr+2q+1, lr+8+2q, lr+9+2q, 8 bytes each from byte 8g: 16-byte chunk
          // g/2 of a 64-byte row, stored at chunk (g/2) ^ ((row >> 1) & 3) = (g/2) ^ q
          // (64-byte swizzle).  Lanes with odd q load the odd row first, so that the 16
          // lanes of each access phase cover all 32 banks once.
          const int rows[4] = {lr + 2 * q, lr + 2 * q + 1, lr + 8 + 2 * q, lr + 9 + 2 * q};
          const uint32_t wbase = smem_u32(ws_w) + static_cast<uint32_t>((((g >> 1) ^ q) << 4) + 8 * (g & 1));
          const int odd = q & 1;
          uint2 w[4];
          {
            const uint32_t ra = wbase + static_cast<uint32_t>(lr + 2 * q + odd) * F::kRowBytes;       // first
            const uint32_t rb = wbase + static_cast<uint32_t>(lr + 2 * q + 1 - odd) * F::kRowBytes;   // second
            const uint2 x0 = lds_u64(ra);
            const uint2 x1 = lds_u64(rb);
            const uint2 x2 = lds_u64(ra + 8 * F::kRowBytes);
            const uint2 x3 = lds_u64(rb + 8 * F::kRowBytes);
            w[0] = odd ? x1 : x0;
            w[1] = odd ? x0 : x1;
            w[2] = odd ? x3 : x2;
            w[3] = odd ? x2 : x3;
          }
          uint32_t sraw[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int grow = n0 + c * kChunk + rows[i];
            if (p.scale_tma) {
              sraw[i] = FMT == BSQ_MXFP4 ? ws_s[rows[i] * 16 + ((cb >> 5) & 15) + (g >> 1)]
                                         : ws_s[rows[i] * 16 + ((cb >> 4) & 15) + g];
            } else {
              sraw[i] = 0;
              if (col_ok && grow < n1)
                sraw[i] = __ldg(scale_e + static_cast<int64_t>(grow) * p.scale_ld + (FMT == BSQ_MXFP4 ? (col >> 5) : (col >> 4)));
            }
          }
          // the scales of the k-step's four rows (rows 2q, 2q+1 pair in b0, rows 8+2q, 9+2q in b1)
          const ScaleBf16 sc0 = pair_scales(row_scale<FMT>(sraw[0], tscale), row_scale<FMT>(sraw[1], tscale));
          const ScaleBf16 sc1 = pair_scales(row_scale<FMT>(sraw[2], tscale), row_scale<FMT>(sraw[3], tscale));
          const bool fast = sc0.fast && sc1.fast;
#pragma unroll
          for (int wi = 0; wi < 2; ++wi) {
            uint32_t b0[8], b1[8];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const uint32_t* xw = reinterpret_cast<const uint32_t*>(&w[2 * half]);
              const uint32_t* yw = reinterpret_cast<const uint32_t*>(&w[2 * half + 1]);
              uint32_t(&dst)[8] = half ? b1 : b0;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint32_t v = pair_bytes(xw[wi], yw[wi], j);                // byte 4wi+j of both rows
                dst[2 * j] = ((v & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;         // column 8wi+2j
                dst[2 * j + 1] = ((v & 0x00F000F0u) * 0x0104u) & 0x81C081C0u;     // column 8wi+2j+1
              }
            }
            if (fast) {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                b0[j] = bf16x2_mul(b0[j], sc0.c2);
                b1[j] = bf16x2_mul(b1[j], sc1.c2);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                b0[j] = scale_one(b0[j], sc0, kPow2_126x2);
                b1[j] = scale_one(b1[j], sc1, kPow2_126x2);
              }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) mma_bf16_16816(acc[8 * wi + j], a, b0[j], b1[j]);
          }
        }
        // This warp is done with the chunk's slot (its reads are in registers and consumed).
        // The fourth warp of the group to let it go refills it with the chunk kRing later:
        // nobody waits for a slot to drain.  Every lane orders its plain reads of the slot
        // before the copy (the async proxy) that overwrites it.
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          const uint32_t prior = atomicAdd(&released[si], 1u);
          if ((prior & 3u) == 3u && c + kRing < nchunks) {
            __threadfence_block();
            fence_proxy_async_smem();
            issue(cc + kRing, c + kRing, e, r0);
          }
        }
      }
      // One decision for the CTA; after a timeout the CTA writes nothing, lets its copies in
      // flight land and still meets its cluster at both barriers.
      ok = __syncthreads_and(ok) != 0;
      if (!ok) {
        if (tid == 0) {
          atomicCAS(p.err, 0, BSQ_DEVERR_TIMEOUT);
          // the last fill of every slot (slot fills are issued in order)
          for (int s = 0; s < kRing; ++s) {
            if (fills[s] == 0) continue;
            const uint64_t w0 = global_timer_ns();
            while (!mbar_try_wait(smem_u32(&full[s]), (fills[s] - 1) & 1) && global_timer_ns() - w0 < kDrainLimitNs) {
            }
          }
        }
        __syncthreads();
      } else {
        // Every warp stores its partial through the idle ring, fragment by fragment
        // ([warp][n-tile][fragment register][lane], conflict-free); then every thread adds the
        // eight warps' values of its entries and writes the CTA's partial red[token][column]
        // (column = 16 n + n-tile of the slab).
        {
          float* dst = tree + warp * (kNT * 4 * 32);
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) dst[(nt * 4 + r) * 32 + lane] = acc[nt][r];
        }
        __syncthreads();
        for (int i = tid; i < kNT * 4 * 32; i += kThreadsSm) {
          float v = 0.f;
#pragma unroll
          for (int w2 = 0; w2 < kWarps; ++w2) v += tree[w2 * (kNT * 4 * 32) + i];
          const int l = i & 31, rr = (i >> 5) & 3, nt = i >> 7;
          const int t = (l >> 2) + ((rr & 2) ? 8 : 0), n = 2 * (l & 3) + (rr & 1);
          red[t * kSlab + 16 * n + nt] = v;
        }
      }
      if (tid == 0) *pass_ok = ok ? 1 : 0;
      // Every partial of the cluster and its status are in place (release/acquire at cluster scope) ...
      cluster_sync();
      {
        uint32_t peer_ok = 1u;
        if (static_cast<uint32_t>(lane) < csize) peer_ok = ld_shared_cluster_u32(map_to_rank(smem_u32(pass_ok), lane));
        live = __all_sync(0xffffffffu, peer_ok != 0u);
      }
      // ... and CTA r of the cluster adds columns [r*cw, (r+1)*cw) of the slab over all of them.
      const int cw = ((kSlab + static_cast<int>(csize) - 1) / static_cast<int>(csize) + 3) & ~3;
      const int c_lo = static_cast<int>(crank) * cw, c_hi = min(kSlab, c_lo + cw);
      if (live && c_hi > c_lo) {
        const int span = c_hi - c_lo;
        for (int i = tid; i < mt * span; i += kThreadsSm) {
          const int t = i / span, cc = c_lo + i % span;
          const uint32_t off = smem_u32(red + t * kSlab + cc);
          float v = 0.f;
          for (uint32_t r = 0; r < csize; ++r) v += ld_shared_cluster_f32(map_to_rank(off, r));
          if (cb + cc < p.K) p.out[static_cast<int64_t>(r0 + t) * p.K + cb + cc] = __float2bfloat16_rn(v);
        }
      }
      // The ring was written as plain shared memory (the warp partials); the next pass's
      // copies write it through the async proxy.
      fence_proxy_async_smem();
      // No CTA goes on (or leaves) while its peers may still read its partial.
      cluster_sync();
      cbase += static_cast<uint32_t>(nchunks);
    }
  }
}

}  // namespace

size_t smallm_workspace_bytes(int64_t K) {
  const int64_t slabs = (K + kSlab - 1) / kSlab;
  return static_cast<size_t>(16 * K * 4 + ((slabs * 4 + 255) / 256) * 256 + 256);
}

int launch_smallm(const SmallMArgs& a, const char** msg) {
  SmallParams p;
  p.scale = static_cast<const uint8_t*>(a.w_scale);
  p.tensor_scale = a.w_tensor_scale;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.M = static_cast<int32_t>(a.M);
  p.N = static_cast<int32_t>(a.N);
  p.K = static_cast<int32_t>(a.K);
  p.err = a.err;
  p.timeout_ns = wait_limit_ns();
  p.scale_ld = a.fmt == BSQ_MXFP4 ? static_cast<int32_t>(a.K / 32)
               : a.fmt == BSQ_NVFP4 ? static_cast<int32_t>(a.K / 16)
                                    : static_cast<int32_t>((a.K + 127) / 128);
  const int slabs = static_cast<int>((a.K + kSlab - 1) / kSlab);
  // about two CTAs per SM in one wave; rows per CTA a multiple of 128, at most 512
  int splits = (2 * a.num_sms) / slabs;
  splits = splits < 1 ? 1 : splits;
  int rps = static_cast<int>((a.N + splits - 1) / splits);
  rps = (rps + kStep * kWarps - 1) / (kStep * kWarps) * (kStep * kWarps);
  if (rps > kMaxRows) rps = kMaxRows;
  splits = static_cast<int>((a.N + rps - 1) / rps);
  p.rows_per_split = rps;
  p.ws = static_cast<float*>(a.ws);
  p.counters = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(a.ws) + static_cast<size_t>(16 * a.K * 4));
  if (splits > 1 && !a.ws) {
    *msg = "small-M dgrad needs a workspace";
    return -1;
  }
  // tensor maps: packed W [N][K(/2)], scales [N][K/32 or K/16], grad_out [M][N]
  CUtensorMap tm_w, tm_s, tm_g;
  const uint64_t wrow = a.fmt == BSQ_FP8_E4M3_B128 ? a.K : a.K / 2;
  {
    const uint64_t dims[2] = {wrow, static_cast<uint64_t>(a.N)};
    const uint64_t strides[1] = {wrow};
    const uint32_t box[2] = {static_cast<uint32_t>(a.fmt == BSQ_FP8_E4M3_B128 ? kSlab : kSlab / 2),
                             static_cast<uint32_t>(kBox)};
    if (!encode_map(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.w_data, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE)) {
      *msg = "tensor map encoding failed for W";
      return -1;
    }
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(a.N) * 2};
    const uint32_t box[2] = {64, 16};
    if (!encode_map(&tm_g, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.g, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) {
      *msg = "tensor map encoding failed for grad_out";
      return -1;
    }
  }
  tm_s = tm_w;
  p.scale_tma = 0;
  if (a.fmt == BSQ_MXFP4 || a.fmt == BSQ_NVFP4) {
    const uint64_t srow = a.fmt == BSQ_MXFP4 ? a.K / 32 : a.K / 16;
    if (srow % 16 == 0 && (reinterpret_cast<uintptr_t>(a.w_scale) & 15u) == 0) {
      const uint64_t dims[2] = {srow, static_cast<uint64_t>(a.N)};
      const uint64_t strides[1] = {srow};
      const uint32_t box[2] = {16, static_cast<uint32_t>(kBox)};
      if (!encode_map(&tm_s, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.w_scale, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_NONE)) {
        *msg = "tensor map encoding failed for the scales";
        return -1;
      }
      p.scale_tma = 1;
    }
  }
  const dim3 grid(slabs, splits);
  cudaError_t e = cudaSuccess;
#define BSQ_LAUNCH_SMALL(F_)                                                                                 \
  e = cudaFuncSetAttribute(smallm_dgrad_kernel<F_>, cudaFuncAttributeMaxDynamicSharedMemorySize,            \
                           SmallFmt<F_>::kSmem);                                                             \
  if (e == cudaSuccess) smallm_dgrad_kernel<F_><<<grid, kThreadsSm, SmallFmt<F_>::kSmem, a.stream>>>(tm_w, tm_s, tm_g, p);
  switch (a.fmt) {
    case BSQ_MXFP4: BSQ_LAUNCH_SMALL(BSQ_MXFP4) break;
    case BSQ_NVFP4: BSQ_LAUNCH_SMALL(BSQ_NVFP4) break;
    case BSQ_FP8_E4M3_B128: BSQ_LAUNCH_SMALL(BSQ_FP8_E4M3_B128) break;
    default:
      *msg = "small-M dgrad: unsupported format";
      return -1;
  }
#undef BSQ_LAUNCH_SMALL
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    *msg = cudaGetErrorString(e);
    return static_cast<int>(e);
  }
  return 0;
}

namespace {
int env_rows(const char* name, int dflt) {
  const char* v = std::getenv(name);
  if (!v || !*v) return dflt;
  const long r = std::strtol(v, nullptr, 10);
  return r < 0 ? 0 : (r > kTileN - 1 ? kTileN - 1 : static_cast<int>(r));
}
}  // namespace

// Shared memory and its carveout for a small-M kernel (the carveout at its maximum, so
// that two CTAs fit on an SM).
template <typename Kern>
static cudaError_t set_smem(Kern kern, int bytes) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  return e;
}

// Clusters of `size` CTAs of the small-M kernel that fit on the current device at once
// (cudaOccupancyMaxActiveClusters), cached per device; 0 when the query fails.
static int resident_clusters(int fmt, int size) {
  static std::mutex mu;
  static int table[kMaxDevices][3][kMaxSplits + 1];
  static bool init = false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  const int fi = fmt == BSQ_MXFP4 ? 0 : fmt == BSQ_NVFP4 ? 1 : 2;
  std::lock_guard<std::mutex> lock(mu);
  if (!init) {
    for (auto& d : table)
      for (auto& f : d)
        for (int& v : f) v = -1;
    init = true;
  }
  int& slot = table[dev][fi][size];
  if (slot >= 0) return slot;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(size);
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(1, static_cast<unsigned>(size), 1);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  cudaError_t e = cudaSuccess;
#define BSQ_OCC(F_)                                                                                  \
  cfg.blockDim = dim3(kThreadsSm);                                                                   \
  cfg.dynamicSmemBytes = ClusterFmt<F_>::kSmem;                                                      \
  e = set_smem(smallm_dgrad_cluster_kernel<F_>, ClusterFmt<F_>::kSmem);                              \
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, smallm_dgrad_cluster_kernel<F_>, &cfg);
  if (fi == 0) {
    BSQ_OCC(BSQ_MXFP4)
  } else if (fi == 1) {
    BSQ_OCC(BSQ_NVFP4)
  } else {
    BSQ_OCC(BSQ_FP8_E4M3_B128)
  }
#undef BSQ_OCC
  if (e != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  slot = n;
  return n;
}

int grouped_small_rows() { return env_rows("BSQ_GROUPED_SMALL_ROWS", kGroupedSmallRows); }
int grouped_tail_rows() { return env_rows("BSQ_GROUPED_TAIL_ROWS", 0); }

int launch_smallm_cluster(const SmallMArgs& a, const char** msg) {
  const int fmt = kernel_fmt(a.fmt);
  const bool grouped = a.offsets != nullptr;
  ClusterParams p;
  p.scale = static_cast<const uint8_t*>(a.w_scale);
  p.tensor_scale = a.w_tensor_scale;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.offsets = a.offsets;
  p.S = static_cast<int32_t>(a.M);
  p.N = static_cast<int32_t>(a.N);
  p.K = static_cast<int32_t>(a.K);
  p.E = grouped ? static_cast<int32_t>(a.E) : 1;
  p.tail_rows = grouped ? a.tail_rows : 0;
  p.err = a.err;
  p.timeout_ns = wait_limit_ns();
  // Test hook (failure detection without a GPU fault): with BSQ_TEST_DROP_CHUNK=1 the first
  // chunk of every CTA is never requested, so the wait for it runs out and the kernel takes
  // its orderly abort.
  const char* drop = std::getenv("BSQ_TEST_DROP_CHUNK");
  p.drop_chunk = drop && drop[0] == '1' ? 1 : 0;
  const bool per_tensor = a.fmt == BSQ_FP8_E4M3_TENSOR;
  p.scale_ld = fmt == BSQ_MXFP4 ? static_cast<int32_t>(a.K / 32)
               : fmt == BSQ_NVFP4 ? static_cast<int32_t>(a.K / 16)
               : per_tensor       ? 1
                                  : static_cast<int32_t>((a.K + 127) / 128);
  p.scale_batch = fmt == BSQ_FP8_E4M3_B128 ? (per_tensor ? 1 : ((a.N + 127) / 128) * p.scale_ld) : a.N * p.scale_ld;
  p.scale_shift = fp8_scale_shift(a.fmt);
  const int slabs = static_cast<int>((a.K + kSlab - 1) / kSlab);
  // Experts walked at once (grid z): every one that can have rows here when the whole
  // grouped product is this kernel's (S within tail_rows), else an estimate of how many
  // ragged last tiles fall within tail_rows; a CTA takes further experts in turn.
  int64_t gz = 1;
  if (grouped) {
    gz = a.M <= a.tail_rows ? std::min<int64_t>(a.E, a.M) : (a.E * a.tail_rows + kTileN - 1) / kTileN;
    gz = std::max<int64_t>(1, std::min<int64_t>(gz, std::min<int64_t>(a.E, a.M)));
  }
  // Row splits = the cluster size, at most 8 and no more than there are 64-row chunks.
  // One weight: fewer clusters of a larger size fit on the GPU at once (a cluster's CTAs
  // share one GPC), so the size is the one with the least time by (waves of resident
  // clusters) x (chunks per split); ties go to fewer splits.  Grouped: most grid-z slots of
  // a decode-sized call hold no expert and end at once, so the grid is sized as if every
  // slot worked, about two CTAs per SM.
  const int64_t max_by_rows = (a.N + kChunk - 1) / kChunk;
  int64_t splits = 1, best = -1;
  if (grouped) {
    splits = std::max<int64_t>(1, std::min<int64_t>({(2 * a.num_sms) / (slabs * gz), kMaxSplits, max_by_rows}));
    best = 0;
  }
  for (int64_t sz = 1; !grouped && sz <= std::min<int64_t>(kMaxSplits, max_by_rows); ++sz) {
    const int act = resident_clusters(fmt, static_cast<int>(sz));
    if (act <= 0) continue;
    const int64_t waves = (slabs * gz + act - 1) / act;
    const int64_t cost = waves * ((a.N + sz * kChunk - 1) / (sz * kChunk));
    if (best < 0 || cost < best) {
      best = cost;
      splits = sz;
    }
  }
  int64_t rps = (a.N + splits - 1) / splits;
  rps = (rps + kChunk - 1) / kChunk * kChunk;
  p.rows_per_split = static_cast<int32_t>(rps);
  const uint64_t batch = static_cast<uint64_t>(p.E);
  CUtensorMap tm_w, tm_s, tm_g;
  const uint64_t wrow = fmt == BSQ_FP8_E4M3_B128 ? a.K : a.K / 2;
  {
    const uint64_t dims[3] = {wrow, static_cast<uint64_t>(a.N), batch};
    const uint64_t strides[2] = {wrow, wrow * static_cast<uint64_t>(a.N)};
    const uint32_t box[3] = {static_cast<uint32_t>(fmt == BSQ_FP8_E4M3_B128 ? kSlab : kSlab / 2),
                             static_cast<uint32_t>(kChunk), 1};
    // rows of 128 (FP8) or 64 (FP4) bytes, swizzled so that the decode's reads are free of
    // bank conflicts
    const CUtensorMapSwizzle sw = fmt == BSQ_FP8_E4M3_B128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (!encode_map(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.w_data, dims, strides, box, sw)) {
      *msg = "tensor map encoding failed for W";
      return -1;
    }
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(a.N) * 2};
    const uint32_t box[2] = {64, kTok};
    if (!encode_map(&tm_g, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.g, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) {
      *msg = "tensor map encoding failed for grad_out";
      return -1;
    }
  }
  tm_s = tm_w;
  p.scale_tma = 0;
  if (fmt == BSQ_MXFP4 || fmt == BSQ_NVFP4) {
    const uint64_t srow = fmt == BSQ_MXFP4 ? a.K / 32 : a.K / 16;
    if (srow % 16 == 0 && (reinterpret_cast<uintptr_t>(a.w_scale) & 15u) == 0) {
      const uint64_t dims[3] = {srow, static_cast<uint64_t>(a.N), batch};
      const uint64_t strides[2] = {srow, srow * static_cast<uint64_t>(a.N)};
      const uint32_t box[3] = {16, static_cast<uint32_t>(kChunk), 1};
      if (!encode_map(&tm_s, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.w_scale, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_NONE)) {
        *msg = "tensor map encoding failed for the scales";
        return -1;
      }
      p.scale_tma = 1;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(splits);
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(slabs), static_cast<unsigned>(splits), static_cast<unsigned>(gz));
  cfg.blockDim = dim3(kThreadsSm);
  cfg.stream = a.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaSuccess;
#define BSQ_LAUNCH_CLUSTER(F_)                                                                                       \
  cfg.dynamicSmemBytes = ClusterFmt<F_>::kSmem;                                                                     \
  e = set_smem(smallm_dgrad_cluster_kernel<F_>, ClusterFmt<F_>::kSmem);                                             \
  if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, smallm_dgrad_cluster_kernel<F_>, tm_w, tm_s, tm_g, p);
  switch (fmt) {
    case BSQ_MXFP4: BSQ_LAUNCH_CLUSTER(BSQ_MXFP4) break;
    case BSQ_NVFP4: BSQ_LAUNCH_CLUSTER(BSQ_NVFP4) break;
    case BSQ_FP8_E4M3_B128: BSQ_LAUNCH_CLUSTER(BSQ_FP8_E4M3_B128) break;
    default:
      *msg = "small-M dgrad: unsupported format";
      return -1;
  }
#undef BSQ_LAUNCH_CLUSTER
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
// allocation after start-up.  bsq_linear_dgrad_smallm_noalloc serves them with the
// split-K small-M kernel above (smallm_dgrad_kernel), its scratch living in this
// file-scope device array.  The array exists on every device that loads the library, for
// the life of the process.
namespace {

constexpr int64_t kStaticMaxK = 16384;  // largest K the static scratch serves
constexpr size_t kStaticScratchBytes = 16 * kStaticMaxK * 4 + 4096;
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevicesStatic = bsq::kMaxDevices;
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
  if (w_fmt == BSQ_BF16 || w_fmt == BSQ_FP8_E4M3_TENSOR)
    return static_cast<bsq_status>(bsq::set_error(
        BSQ_ERR_UNSUPPORTED, "bsq_linear_dgrad_smallm_noalloc: W must be FP8 (128x128 blocks), MXFP4 or NVFP4"));
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
  int32_t* errw = nullptr;
  int sms2 = 0;
  const int st2 = bsq::device_error_word(&errw, &sms2);
  if (st2 != BSQ_OK) return static_cast<bsq_status>(st2);
  bsq::SmallMArgs a{w_fmt, grad_out, w_data, w_scale, w_tensor_scale, M, N, K, grad_x, scratch, sms, s, errw};
  const char* msg = "";
  if (bsq::launch_smallm(a, &msg) != 0) return static_cast<bsq_status>(bsq::set_error(BSQ_ERR_CUDA, msg));
  return BSQ_OK;
}

