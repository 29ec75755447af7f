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
#include <cstdio>
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
// The same product without any global workspace: the CTAs that split a column slab's rows
// form one thread-block cluster and add their partial sums through distributed shared
// memory.  Each CTA streams its rows in 64-row chunks, each chunk on its own barrier, so
// decoding starts with the first chunk instead of after the whole slab.
constexpr int kChunk = 64;        // rows of W per TMA chunk (four mma k-steps)
constexpr int kRing = 8;          // chunks in flight per CTA
constexpr int kMaxSplits = 8;     // CTAs of a cluster (portable cluster size)

struct ClusterParams {
  const uint8_t* scale;
  const float* tensor_scale;
  __nv_bfloat16* out;
  int32_t M, N, K;
  int32_t rows_per_split;   // multiple of kChunk
  int32_t scale_ld;         // MXFP4: K/32, NVFP4: K/16, FP8: ceil(K/128) (1 with one scale per tensor)
  int32_t scale_shift;      // FP8: log2 of the scale block's side (7; 31 for one scale per tensor)
  int32_t scale_tma;        // FP4 scale windows through TMA
  uint64_t timeout_ns;
  int32_t* err;
};

template <int FMT>
struct ClusterFmt {
  static constexpr int kRowBytes = FMT == BSQ_FP8_E4M3_B128 ? kSlab : kSlab / 2;
  static constexpr int kWBytes = kChunk * kRowBytes;
  static constexpr int kSBytes = FMT == BSQ_FP8_E4M3_B128 ? 0 : kChunk * 16;
  static constexpr int kGBytes = 16 * kChunk * 2;   // [16 tokens][64 rows] BF16, 128-byte swizzled
  static constexpr int kSlotBytes = kWBytes + kSBytes + kGBytes;
  static_assert(kSlotBytes % 1024 == 0, "swizzled grad_out boxes need 1024-byte aligned slots");
  static constexpr int kRingBytes = kRing * kSlotBytes;
  static constexpr int kTreeBytes = kWarps * 16 * kSlab * 4;   // partials of the eight warps
  static constexpr int kStaged = kRingBytes > kTreeBytes ? kRingBytes : kTreeBytes;
  static constexpr int kRedBytes = 16 * kSlab * 4;        // this CTA's partial, read by the cluster
  static constexpr int kSmem = kStaged + kRedBytes + 256 + 1024;
};

template <int FMT>
__global__ void __launch_bounds__(kThreadsSm, 2)
    smallm_dgrad_cluster_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s,
                                const __grid_constant__ CUtensorMap tm_g, const ClusterParams p) {
  using F = ClusterFmt<FMT>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* tree = reinterpret_cast<float*>(base);                  // warp partials; reuse the ring after the last chunk
  float* red = reinterpret_cast<float*>(base + F::kStaged);      // [16 tokens][128 columns]
  uint64_t* full = reinterpret_cast<uint64_t*>(base + F::kStaged + F::kRedBytes);
  uint64_t* empty = full + kRing;
  int32_t* fills = reinterpret_cast<int32_t*>(empty + kRing);   // copies issued into each slot
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

  auto slot_of = [&](int c) { return base + (c % kRing) * F::kSlotBytes; };
  auto issue = [&](int c) {          // TMA of chunk c into its ring slot
    uint8_t* s = slot_of(c);
    fills[c % kRing] += 1;
    const uint32_t bar = smem_u32(&full[c % kRing]);
    const int row = n0 + c * kChunk;
    mbar_arrive_expect_tx(bar, F::kWBytes + ((F::kSBytes && p.scale_tma) ? F::kSBytes : 0) + F::kGBytes);
    tma_load_2d(smem_u32(s), &tm_w, bar, FMT == BSQ_FP8_E4M3_B128 ? cb : cb / 2, row);
    if (F::kSBytes && p.scale_tma)
      tma_load_2d(smem_u32(s + F::kWBytes), &tm_s, bar, (FMT == BSQ_MXFP4 ? (cb >> 5) : (cb >> 4)) & ~15, row);
    tma_load_2d(smem_u32(s + F::kWBytes + F::kSBytes), &tm_g, bar, row, 0);
  };
  if (tid == 0) {
    for (int s = 0; s < kRing; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 4);   // the four warps of the chunk's group
      fills[s] = 0;
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int c = 0; c < min(nchunks, kRing); ++c) issue(c);

  float tscale = 0.f;
  if (FMT == BSQ_NVFP4) tscale = __ldg(p.tensor_scale);
  const int col = cb + 16 * g;
  const bool col_ok = col < p.K;
  float acc[kNT][4];
#pragma unroll
  for (int i = 0; i < kNT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  bool ok = true;
  for (int c = grp; c < nchunks; c += 2) {
    const int si = c % kRing;
    const uint32_t par = (c / kRing) & 1u;
    {
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait_sleep(smem_u32(&full[si]), par, 20000u)) {
        if (global_timer_ns() - t0 > p.timeout_ns) {
          ok = false;
          break;
        }
      }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    const uint8_t* ws_w = slot_of(c);
    const uint8_t* ws_s = ws_w + F::kWBytes;
    const uint32_t gb = smem_u32(ws_w + F::kWBytes + F::kSBytes);
    const int lr = kstep * kStep;                 // the k-step's first row inside the chunk
    const int grow0 = n0 + c * kChunk + lr;       // its row of W
    const int rows[4] = {lr + 2 * q, lr + 2 * q + 1, lr + 8 + 2 * q, lr + 9 + 2 * q};
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
      float sf = 0.f;
      if (col_ok && grow0 < n1)
        sf = __ldg(reinterpret_cast<const float*>(p.scale) + static_cast<int64_t>(grow0 >> p.scale_shift) * p.scale_ld +
                   (col >> p.scale_shift));
      const ScaleBf16 sc = make_scale_fp8(sf);   // one scale block holds the whole k-step
      uint4 w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = *reinterpret_cast<const uint4*>(ws_w + rows[i] * F::kRowBytes + 16 * g);
      const bool any_nan = e4m3_any_nan(w[0].x | w[0].y | w[0].z | w[0].w | w[1].x | w[1].y | w[1].z | w[1].w |
                                        w[2].x | w[2].y | w[2].z | w[2].w | w[3].x | w[3].y | w[3].z | w[3].w);
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
      uint2 w[4];
      uint32_t sraw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        w[i] = *reinterpret_cast<const uint2*>(ws_w + rows[i] * F::kRowBytes + 8 * g);
        const int grow = n0 + c * kChunk + rows[i];
        if (p.scale_tma) {
          sraw[i] = FMT == BSQ_MXFP4 ? ws_s[rows[i] * 16 + ((cb >> 5) & 15) + (g >> 1)]
                                     : ws_s[rows[i] * 16 + ((cb >> 4) & 15) + g];
        } else {
          sraw[i] = 0;
          if (col_ok && grow < n1)
            sraw[i] = __ldg(p.scale + static_cast<int64_t>(grow) * p.scale_ld + (FMT == BSQ_MXFP4 ? (col >> 5) : (col >> 4)));
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
    // this warp is done with the chunk's slot; the group's first warp refills it with the
    // chunk kRing later once all four have let it go
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[si]));
    if (kstep == 0 && lane == 0 && c + kRing < nchunks) {
      const uint64_t t0 = global_timer_ns();
      bool freed = true;
      while (!mbar_try_wait(smem_u32(&empty[si]), par)) {
        if (global_timer_ns() - t0 > p.timeout_ns) {
          freed = false;
          break;
        }
      }
      if (freed) issue(c + kRing);
      else ok = false;
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
  }
  // One decision for the CTA; after a timeout the CTA writes nothing but still meets its
  // cluster at both barriers (its peers read its partial, which is then undefined).
  ok = __syncthreads_and(ok) != 0;
  if (!ok) {
    if (tid == 0) {
      atomicCAS(p.err, 0, BSQ_DEVERR_TIMEOUT);
      // let the copies still in flight land before the shared memory is reused or freed:
      // the last fill of every slot (slot fills are issued in order)
      for (int s = 0; s < kRing; ++s) {
        if (fills[s] == 0) continue;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(smem_u32(&full[s]), (fills[s] - 1) & 1) && global_timer_ns() - t0 < kDrainLimitNs) {
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
    for (int e = tid; e < kNT * 4 * 32; e += kThreadsSm) {
      float v = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < kWarps; ++w2) v += tree[w2 * (kNT * 4 * 32) + e];
      const int l = e & 31, rr = (e >> 5) & 3, nt = e >> 7;
      const int t = (l >> 2) + ((rr & 2) ? 8 : 0), n = 2 * (l & 3) + (rr & 1);
      red[t * kSlab + 16 * n + nt] = v;
    }
  }
  // Every partial of the cluster is in place (release/acquire at cluster scope) ...
  cluster_sync();
  // ... and CTA r of the cluster adds columns [r*cw, (r+1)*cw) of the slab over all of them.
  const int cw = ((kSlab + static_cast<int>(csize) - 1) / static_cast<int>(csize) + 3) & ~3;
  const int c_lo = static_cast<int>(crank) * cw, c_hi = min(kSlab, c_lo + cw);
  if (ok && c_hi > c_lo) {
    const int span = c_hi - c_lo;
    for (int i = tid; i < p.M * span; i += kThreadsSm) {
      const int t = i / span, cc = c_lo + i % span;
      const uint32_t off = smem_u32(red + t * kSlab + cc);
      float v = 0.f;
      for (uint32_t r = 0; r < csize; ++r) v += ld_shared_cluster_f32(map_to_rank(off, r));
      if (cb + cc < p.K) p.out[static_cast<int64_t>(t) * p.K + cb + cc] = __float2bfloat16_rn(v);
    }
  }
  // No CTA leaves while its peers may still read its partial.
  cluster_sync();
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

int launch_smallm_cluster(const SmallMArgs& a, const char** msg) {
  const int fmt = kernel_fmt(a.fmt);
  ClusterParams p;
  p.scale = static_cast<const uint8_t*>(a.w_scale);
  p.tensor_scale = a.w_tensor_scale;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.M = static_cast<int32_t>(a.M);
  p.N = static_cast<int32_t>(a.N);
  p.K = static_cast<int32_t>(a.K);
  p.err = a.err;
  p.timeout_ns = wait_limit_ns();
  p.scale_ld = fmt == BSQ_MXFP4 ? static_cast<int32_t>(a.K / 32)
               : fmt == BSQ_NVFP4 ? static_cast<int32_t>(a.K / 16)
               : a.fmt == BSQ_FP8_E4M3_TENSOR ? 1
                                  : static_cast<int32_t>((a.K + 127) / 128);
  p.scale_shift = fp8_scale_shift(a.fmt);
  const int slabs = static_cast<int>((a.K + kSlab - 1) / kSlab);
  // Row splits = the cluster size: about two CTAs per SM in one wave, at most 8, and no
  // more splits than 64-row chunks.
  int splits = (2 * a.num_sms) / slabs;
  const int64_t max_by_rows = (a.N + kChunk - 1) / kChunk;
  if (splits > kMaxSplits) splits = kMaxSplits;
  if (splits > max_by_rows) splits = static_cast<int>(max_by_rows);
  if (splits < 1) splits = 1;
  int64_t rps = (a.N + splits - 1) / splits;
  rps = (rps + kChunk - 1) / kChunk * kChunk;
  p.rows_per_split = static_cast<int32_t>(rps);
  CUtensorMap tm_w, tm_s, tm_g;
  const uint64_t wrow = fmt == BSQ_FP8_E4M3_B128 ? a.K : a.K / 2;
  {
    const uint64_t dims[2] = {wrow, static_cast<uint64_t>(a.N)};
    const uint64_t strides[1] = {wrow};
    const uint32_t box[2] = {static_cast<uint32_t>(fmt == BSQ_FP8_E4M3_B128 ? kSlab : kSlab / 2),
                             static_cast<uint32_t>(kChunk)};
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
  if (fmt == BSQ_MXFP4 || fmt == BSQ_NVFP4) {
    const uint64_t srow = fmt == BSQ_MXFP4 ? a.K / 32 : a.K / 16;
    if (srow % 16 == 0 && (reinterpret_cast<uintptr_t>(a.w_scale) & 15u) == 0) {
      const uint64_t dims[2] = {srow, static_cast<uint64_t>(a.N)};
      const uint64_t strides[1] = {srow};
      const uint32_t box[2] = {16, static_cast<uint32_t>(kChunk)};
      if (!encode_map(&tm_s, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.w_scale, dims, strides, box,
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
  cfg.gridDim = dim3(static_cast<unsigned>(slabs), static_cast<unsigned>(splits));
  cfg.blockDim = dim3(kThreadsSm);
  cfg.stream = a.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaSuccess;
#define BSQ_LAUNCH_CLUSTER(F_)                                                                                       \
  cfg.dynamicSmemBytes = ClusterFmt<F_>::kSmem;                                                                     \
  e = cudaFuncSetAttribute(smallm_dgrad_cluster_kernel<F_>, cudaFuncAttributeMaxDynamicSharedMemorySize,           \
                           ClusterFmt<F_>::kSmem);                                                                  \
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

