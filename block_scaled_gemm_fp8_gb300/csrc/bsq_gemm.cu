// bsq_gemm.cu -- fused dequantize + BF16 tensor-core GEMM for the backward pass of a
// block-scaled linear layer and of its grouped (mixture-of-experts) form.
//
//   dgrad  grad_X[S,K]   = grad_out[S,N]   @ deq(W[e])[N,K]     per expert rows
//   wgrad  grad_W[e][N,K] = grad_out[r,N]^T @ deq(X)[r,K]        r = the expert's rows
// (MSLK PR #393 "Implementation Method"; transformers PR #50031
//  `FP8LinearFunction.backward`, `FP8GroupedMatmulFunction.backward`.)
//
// Both products are computed transposed, with the dequantized operand on the M side:
//   D[m = column of the packed operand, n] = sum_k deq(P)[k, m] * G-side[k, n]
// where P is W[e] (k = N index, n = token) for dgrad and X (k = token, n = N index)
// for wgrad.  The packed operand is row-major with m contiguous, so it is an
// "MN-major" A operand: no transpose kernel is needed on either side, and the
// dequantization work per tensor-core FLOP is that of a 128-row operand.
//
// The tensor-core work runs on CTA pairs (clusters of two SMs) with the 2-SM MMA
// (tcgen05.mma.cta_group::2): one pair tile is 256 m x 256 n.  Each CTA dequantizes its
// own 128 m-rows and stages half of the grad_out tile (n rows [r*Nm/2, (r+1)*Nm/2) for
// CTA r and an MMA of width Nm); the MMA reads A and B out of both CTAs' shared memory
// and leaves each CTA's 128 x 256 FP32 accumulator in its own TMEM.  Halving the grad_out
// bytes each SM stages halves the L2->SM traffic per FLOP and the shared memory needed to
// keep the TMA round trip (over a microsecond) covered.
//
// Per CTA (one per SM), 24 warps (default kernel; see Roles for the short-tile one):
//   warp 0      TMA producer of the packed ring: packed tiles and FP4 scale tiles
//   warp 2      allocates / frees TMEM; one lane relays "operand ready" to the even CTA
//   warp 3      TMA producer of the grad_out ring: this CTA's half of the unit's tiles
//   warp 1      MMA issuer, one thread of the even CTA: 4 x (256 x Nm x 16) per k-block
//   warps 4-7   epilogue: tcgen05.ld (16 columns at a time, each load waited for in the
//               same statement) -> BF16 -> global, one TMEM lane quarter each; the FP4
//               short-tile kernel stages each chunk in shared memory for a TMA store
//   warps 8-23  dequantization, two teams of 8 warps; team t takes k-block t of every
//               unit: packed codes (smem) -> BF16, written in the 128-byte swizzled
//               MN-major layout the tensor core reads; also zero the rows of a k-block
//               that lie outside the current expert (wgrad)
// Three rings decouple the chains: the packed ring feeds the dequant teams (plain loads,
// fenced against the async proxy before each slot goes back to its TMA producer); the
// BF16 operand ring feeds the MMA from the dequant teams; the grad_out ring feeds the MMA
// straight from TMA.  All three move in units of two k-blocks, and every barrier phase
// of a ring is waited on by the same threads in unit order (a parity wait cannot then
// mistake a phase two laps away for its own).  The operand and grad_out rings share
// their "slot free" barrier, so the single MMA thread handles one wait, eight MMAs and
// one commit per unit.
// Operand-ready protocol.  The pair MMA issued by the even CTA reads shared memory of
// both CTAs, so what the odd CTA wrote for a unit must be released at cluster scope to
// the issuing thread.  Every dequant warp arrives on its own CTA's a_local barrier once
// its A rows (and any grad_out rows it zeroed) are written and fenced to the async
// proxy; one relay thread per CTA waits for a_local and for the CTA's grad_out half (TMA
// bytes).  The even relay then arrives on a_full expecting 4 transaction bytes; the odd
// relay supplies them with an st.async into the even CTA whose complete-tx is a release
// at cluster scope.  The MMA thread acquires a_full at cluster scope.  (An
// mbarrier.arrive.release.cluster there stalls the SM and costs about 30 % of the
// throughput; the st.async costs next to nothing.)  MMA completion is multicast to both
// CTAs' "slot free" barriers; the odd CTA's epilogue hands TMEM back the same way as the
// odd relay.  Two TMEM accumulators (2 x 256 columns) let the epilogue of one tile
// overlap the main loop of the next.  Tiles are walked in a static persistent order;
// each role finds a tile's expert with its own forward cursor over the offsets (read
// through the read-only cache, so no table takes shared memory).  Every wait is
// bounded by %globaltimer and records a timeout in the device error word (and stops the
// peer CTA) instead of hanging.
#include <atomic>
#include <cstdlib>
#include <type_traits>

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "bsq_decode.cuh"
#include "bsq_internal.h"
#include "bsq_pipe.cuh"
#include "bsq_ptx.cuh"
#include "../../include/bsq.h"

namespace bsq {

namespace {

constexpr int kDeqTeams = 2;                    // dequant team t fills k-block t of every unit
constexpr int kThreads = 768;                    // 4 control warps, epilogue and dequant warps

// Warp roles.  The default kernel has 4 epilogue warps (one per TMEM lane quarter) and two
// dequant teams of 8 warps, each thread decoding one row of its team's k-block.  The
// short-tile kernel (grouped wgrad with few rows per expert, where a tile has a handful of
// k-blocks and its epilogue sets the pace) has 12 epilogue warps, three per lane quarter
// splitting the columns, and two teams of 4 dequant warps decoding two rows per thread.
template <bool SHORT>
struct Roles {
  static constexpr int kEpiWarps = SHORT ? 12 : 4;
  static constexpr int kEpiPerQuarter = kEpiWarps / 4;
  static constexpr int kDeqPerTeam = SHORT ? 4 : 8;
  static constexpr int kRows = 8 / kDeqPerTeam;        // k-block rows decoded per dequant thread
  static constexpr int kRowStep = 8 * kDeqPerTeam;     // distance between a thread's rows
  static constexpr int kFirstDeq = 4 + kEpiWarps;
  static_assert(kFirstDeq + kDeqTeams * kDeqPerTeam == kThreads / 32, "every warp has a role");
};
constexpr int kBoxBytes = 64 * 64 * 2;          // one 64x64 BF16 box = one swizzle column of 64 rows
constexpr int kABytes = kTileM * kTileK * 2;     // 16 KB: dequantized operand, 2 swizzle columns
constexpr int kPair = 2;                         // CTAs of one 2-SM MMA (a cluster)
constexpr uint16_t kPairMask = 3;                // both CTAs of the pair
constexpr int kBHalf = kTileN / kPair;           // grad_out rows (n) staged by each CTA
constexpr int kBBytes = kBHalf * kTileK * 2;     // 16 KB: this CTA's half of the grad_out tile
constexpr int kTmemCols = 512;                   // 2 accumulators x 256 FP32 columns
// The operand and grad_out rings move in units of two k-blocks: one "operand ready"
// barrier, one MMA-completion commit and one grad_out barrier per unit.
constexpr int kUnitKb = 2;
constexpr int kAUnitBytes = kUnitKb * kABytes;   // 32 KB
constexpr int kBUnitBytes = kUnitKb * kBBytes;   // 32 KB
constexpr int kUStages = 3;
static_assert(kUStages >= 2, "the MMA issuer awaits the next unit before committing the current one");
static_assert(kDeqTeams == kUnitKb, "dequant team t fills k-block t of every unit");
constexpr int kMaxStages = 8;

template <int FMT, bool SHORT = false>
struct Fmt {
  static constexpr bool kFp4 = FMT == BSQ_MXFP4 || FMT == BSQ_NVFP4;
  // packed tile of one k-block (BF16: the operand tile itself, already swizzled by TMA)
  static constexpr int kPBytes = FMT == BSQ_FP8_E4M3_B128 ? kTileK * kTileM
                                 : FMT == BSQ_BF16       ? kABytes
                                                         : kTileK * kTileM / 2;
  static constexpr int kPRowBytes = FMT == BSQ_FP8_E4M3_B128 ? kTileM : kTileM / 2;
  // FP4 scale tile staged by TMA: 64 rows x 16 bytes (a 16-byte aligned window of the row's scales)
  static constexpr int kSBytes = kFp4 ? kTileK * 16 : 0;
  static constexpr int kPStageBytes = (kPBytes + kSBytes + 1023) / 1024 * 1024;   // one k-block
  static constexpr int kPUnitBytes = kUnitKb * kPStageBytes;
  // Units of the packed ring.  Like the other rings it moves in units that both dequant
  // teams consume in order, so no parity wait can alias a phase two laps away.
  // The short-tile kernel of an FP4 format stages each epilogue warp's 16 x 32 output
  // chunk in shared memory for a TMA store, paid for with one packed unit.
  static constexpr bool kEpiStaged = SHORT && kFp4;
  static constexpr int kPUnits = (FMT == BSQ_BF16 ? 1 : (FMT == BSQ_FP8_E4M3_B128 ? 2 : 3)) - (kEpiStaged ? 1 : 0);
  static constexpr int kEpiStage = 1024;                                 // [16 n][32 m] BF16 per epilogue warp
  static constexpr int kEpiBytes = kEpiStaged ? Roles<true>::kEpiWarps * kEpiStage : 0;
  static constexpr int kRingBytes = kUStages * (kBUnitBytes + kAUnitBytes) + kPUnits * kPUnitBytes + kEpiBytes;
};

struct Params {
  const uint8_t* scale;
  const float* tensor_scale;
  const int32_t* offsets;
  __nv_bfloat16* out;
  int32_t* err;
  int64_t out_expert_stride;  // wgrad: N*K; dgrad: 0
  int64_t p_rows;             // packed rows per batch entry
  int32_t E;
  int32_t S;
  int32_t N;
  int32_t Kc;
  int32_t num_m;              // ceil(Kc / 128)
  int32_t num_mg;             // ceil(num_m / 2): m-tile pairs, one per pair tile
  int32_t scale_ld;           // scale row pitch (elements)
  int32_t scale_rblocks;      // FP8: scale rows per batch entry (ceil(p_rows / 128), or 1 per tensor)
  int32_t scale_shift;        // FP8: log2 of the scale block's side (7; 31 for one scale per tensor)
  int32_t scale_tma;          // FP4: scale tiles come through TMA (row pitch a multiple of 16 bytes)
  int32_t b_mode;             // grad_out half tile per k-block: 0 = two 64x64 boxes, 1 = one 2-D box, 2 = one 3-D box
  int32_t b_rows;             // mode 1: rows of the box (tokens); mode 2: 64-column atoms in the box
  uint64_t timeout_ns;
  int32_t drop_announce;      // test hook: the even CTA's relay never announces a unit
  int32_t tail_rows;          // grouped dgrad: an expert's last (rows % kTileN) rows, when at most
                              // this many, are left to the small-M kernel (0: none)
};

struct SharedTail {
  uint64_t p_full[kMaxStages];    // per unit: the packed tiles landed (TMA bytes)
  uint64_t p_empty[kMaxStages];   // per unit: every dequant warp of this CTA has read its half
  uint64_t a_local[kMaxStages];   // per unit: this CTA's dequant warps wrote their A rows
  uint64_t a_full[kMaxStages];    // per unit (even CTA's is used): even relay + 4 bytes from the odd relay
  uint64_t op_empty[kMaxStages];  // per unit: the unit's MMAs completed (frees its A and B slots)
  uint64_t b_full[kMaxStages];    // per unit: this CTA's grad_out half landed (TMA bytes)
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t sink;                  // target of the odd CTA's st.async announcements (never read)
  uint32_t abort_flag;
  int32_t total_tiles;
  int32_t first_tiles;             // tiles of the first GEMM of the launch
};

struct TileInfo {
  int e, mt, nt, n_valid, kblocks, r0, r1;
};

// Pair tiles of an expert with cnt rows, and one past the last row of expert e (the
// cumulative end offset; a null offsets pointer is one group of S rows).
// Rows of an expert's dgrad that the pair tiles take: all of them, less a ragged last tile
// of 1..tail_rows rows (the small-M kernel's share; the same rule is applied there).
__device__ __forceinline__ int dgrad_tile_rows(const Params& p, int cnt) {
  const int tail = cnt % kTileN;
  return (tail > 0 && tail <= p.tail_rows) ? cnt - tail : cnt;
}
template <int OP>
__device__ __forceinline__ int expert_tiles(const Params& p, int cnt) {
  const int ntiles = OP == kDgrad ? (dgrad_tile_rows(p, cnt) + kTileN - 1) / kTileN : (p.N + kTileN - 1) / kTileN;
  return ntiles * p.num_mg;
}
__device__ __forceinline__ int expert_end(const Params& p, int e) { return p.offsets ? __ldg(p.offsets + e) : p.S; }

// Each role walks the tiles in the same increasing order and keeps its own cursor over the
// experts: tiles [pre, next) belong to expert e, whose rows are [r0, r1).
struct ExpertCursor {
  int e, pre, next, r0, r1;
};
template <int OP>
__device__ __forceinline__ ExpertCursor cursor_begin(const Params& p) {
  ExpertCursor c;
  c.e = 0;
  c.pre = 0;
  c.r0 = 0;
  c.r1 = expert_end(p, 0);
  c.next = expert_tiles<OP>(p, c.r1);
  return c;
}

template <int OP>
__device__ __forceinline__ TileInfo decode_tile(int t, ExpertCursor& c, const Params& p, int rank) {
  while (c.next <= t) {   // t < total tiles, so this stops at an expert below E
    ++c.e;
    c.pre = c.next;
    c.r0 = c.r1;
    c.r1 = expert_end(p, c.e);
    c.next = c.pre + expert_tiles<OP>(p, c.r1 - c.r0);
  }
  TileInfo ti;
  const int local = t - c.pre;
  ti.e = c.e;
  ti.mt = (local % p.num_mg) * kPair + rank;   // may be past the last m-tile (odd CTA of the last pair)
  ti.nt = local / p.num_mg;
  ti.r0 = c.r0;
  ti.r1 = c.r1;
  const int cnt = ti.r1 - ti.r0;
  if (OP == kDgrad) {
    ti.n_valid = min(kTileN, dgrad_tile_rows(p, cnt) - ti.nt * kTileN);
    ti.kblocks = (p.N + kTileK - 1) / kTileK;
  } else {
    ti.n_valid = min(kTileN, p.N - ti.nt * kTileN);
    ti.kblocks = (cnt + kTileK - 1) / kTileK;
  }
  return ti;
}

// Width of the pair MMA for a tile with n_valid columns.  CTA r stages grad_out n rows
// [r*Nm/2, (r+1)*Nm/2); the 3-D grad_out box (wgrad, b_mode 2) needs Nm/2 to be a whole
// number of 64-column swizzle atoms.
__device__ __forceinline__ int mma_width(bool dgrad, int n_valid, int b_mode) {
  if (!dgrad && b_mode == 2) return n_valid > 128 ? 256 : 128;
  return max(32, (n_valid + 15) & ~15);
}


// This thread's 32 packed codes of one k-block row (FP8: wa = codes 0..15 as read, wb the
// other 16; FP4: wa) -> 4 groups of 4 BF16 pairs, scaled; zeros outside the operand.
template <int FMT>
__device__ __forceinline__ void decode_row(const uint4& wa, const uint4& wb, uint32_t sraw, float sf, float tscale,
                                           bool valid, uint32_t (&v)[4][4]) {
  if (!valid) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) v[j][i] = 0u;
    return;
  }
  if (FMT == BSQ_MXFP4 || FMT == BSQ_NVFP4) {
    spread_e2m1x8(wa.x, v[0]);
    spread_e2m1x8(wa.y, v[1]);
    spread_e2m1x8(wa.z, v[2]);
    spread_e2m1x8(wa.w, v[3]);
    ScaleBf16 s0, s1;
    if (FMT == BSQ_MXFP4) {
      s0 = make_scale_e8m0(sraw);
      s1 = s0;
    } else {
      s0 = make_scale_nvfp4(sraw & 0xFFu, tscale);
      s1 = make_scale_nvfp4(sraw >> 8, tscale);
    }
    if (s0.fast && s1.fast) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[0][i] = bf16x2_mul(v[0][i], s0.c2);
        v[1][i] = bf16x2_mul(v[1][i], s0.c2);
        v[2][i] = bf16x2_mul(v[2][i], s1.c2);
        v[3][i] = bf16x2_mul(v[3][i], s1.c2);
      }
    } else {
      scale_pairs4(v[0], s0, kPow2_126x2);
      scale_pairs4(v[1], s0, kPow2_126x2);
      scale_pairs4(v[2], s1, kPow2_126x2);
      scale_pairs4(v[3], s1, kPow2_126x2);
    }
  } else if (FMT == BSQ_FP8_E4M3_B128) {
    decode_e4m3x32(wa, wb, make_scale_fp8(sf), v);
  }
}

// One GEMM of a launch: its tensor maps (packed operand, grad_out, FP4 scale tiles) and
// parameters (host side; the kernel takes them as separate arguments).
struct OpArgs {
  CUtensorMap tm_p;
  CUtensorMap tm_g;
  CUtensorMap tm_s;
  CUtensorMap tm_o;
  Params p;
};

// Tile t of a launch: whether it belongs to the second GEMM (kBoth) and its coordinates;
// each role keeps its own expert cursors (c0 over the first GEMM's tiles, c1 the second's).
template <int OPS>
__device__ __forceinline__ TileInfo tile_at(int t, int n_first, ExpertCursor& c0, ExpertCursor& c1, const Params& p0,
                                            const Params& p1, int rank, bool& second) {
  second = OPS == kBoth && t >= n_first;
  if (second) return decode_tile<kWgrad>(t - n_first, c1, p1, rank);
  return decode_tile<OPS == kBoth ? static_cast<int>(kDgrad) : OPS>(t, c0, p0, rank);
}

template <typename T>
__device__ __forceinline__ T pick(bool second, T first_value, T second_value) {
  return second ? second_value : first_value;
}

// One launch runs the tiles of one GEMM (OPS = kDgrad or kWgrad, described by a0) or of two
// (OPS = kBoth: the dgrad tiles of a0, then the wgrad tiles of a1, over the same grad_out,
// packed operands of one format and the same expert offsets).  Every role walks the same
// tile sequence; `second` marks a tile of a1.
template <int FMT, int OPS, bool SHORT>
__global__ void __launch_bounds__(kThreads, 1)
    bsq_gemm_kernel(const __grid_constant__ CUtensorMap tm_p0, const __grid_constant__ CUtensorMap tm_g0,
                    const __grid_constant__ CUtensorMap tm_s0, const __grid_constant__ CUtensorMap tm_p1,
                    const __grid_constant__ CUtensorMap tm_g1, const __grid_constant__ CUtensorMap tm_s1,
                    const __grid_constant__ CUtensorMap tm_o, const Params p, const Params p1) {
  using F = Fmt<FMT, SHORT>;
  using R = Roles<SHORT>;
  constexpr int OP0 = OPS == kBoth ? static_cast<int>(kDgrad) : OPS;
  static_assert(!SHORT || FMT != BSQ_BF16, "the short-tile kernel decodes packed formats only");
  static_assert(!SHORT || OPS == kWgrad, "the short-tile kernel runs wgrad launches only");
  // p: the first GEMM, and the fields both GEMMs share (offsets, E, S, N, Kc, tiling, error
  // word, wait limit); p1: the second GEMM of a kBoth launch.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring_b = smem;
  uint8_t* ring_a = ring_b + kUStages * kBUnitBytes;
  uint8_t* ring_p = ring_a + kUStages * kAUnitBytes;
  uint8_t* ring_e = ring_p + F::kPUnits * F::kPUnitBytes;
  SharedTail& sh = *reinterpret_cast<SharedTail*>(smem + F::kRingBytes);
  volatile uint32_t* abort_flag = &sh.abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---------------------------------------------------------------- set-up
  if (tid == 0) {
    for (int s = 0; s < F::kPUnits; ++s) {
      mbar_init(smem_u32(&sh.p_full[s]), 1);
      mbar_init(smem_u32(&sh.p_empty[s]), R::kDeqPerTeam * kDeqTeams);   // every dequant warp of this CTA
    }
    for (int s = 0; s < kUStages; ++s) {
      mbar_init(smem_u32(&sh.a_local[s]), R::kDeqPerTeam * kDeqTeams);   // every dequant warp of this CTA
      mbar_init(smem_u32(&sh.a_full[s]), 1);                             // even relay; odd relay: tx bytes
      mbar_init(smem_u32(&sh.op_empty[s]), 1);
      mbar_init(smem_u32(&sh.b_full[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sh.tmem_full[b]), 1);
      mbar_init(smem_u32(&sh.tmem_empty[b]), R::kEpiWarps);   // even epilogue warps; odd ones: tx bytes
    }
    mbar_init(smem_u32(&sh.drain), 1);
    sh.abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tm_p0);
    tma_prefetch_map(&tm_g0);
    if (F::kFp4 && p.scale_tma) tma_prefetch_map(&tm_s0);
    if (OPS == kBoth) {
      tma_prefetch_map(&tm_p1);
      tma_prefetch_map(&tm_g1);
      if (F::kFp4 && p1.scale_tma) tma_prefetch_map(&tm_s1);
    }
  }
  if (warp == 2) {
    tmem_alloc_pair(smem_u32(&sh.tmem_base), kTmemCols);
    tmem_relinquish_pair();
  }
  const int E = p.E;
  if (warp == 3) {
    // Validate the offsets and count the tiles: lane l owns experts [l*per, (l+1)*per).
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int bad = 0, sum0 = 0, sum1 = 0;
    int a = e0 == 0 ? 0 : expert_end(p, e0 - 1);
    for (int e = e0; e < e1; ++e) {
      const int b = expert_end(p, e);
      if (b < a || b > p.S || a < 0) bad = 1;
      sum0 += expert_tiles<OP0>(p, max(b - a, 0));
      if (OPS == kBoth) sum1 += expert_tiles<kWgrad>(p1, max(b - a, 0));
      a = b;
    }
    bad = __any_sync(0xffffffffu, bad);
    const int t0 = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(sum0)));
    const int t1 = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(sum1)));
    if (lane == 0) {
      sh.total_tiles = bad ? 0 : t0 + t1;
      sh.first_tiles = t0;
      if (bad && blockIdx.x == 0) record_error(p.err, BSQ_DEVERR_BAD_OFFSETS);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();   // both CTAs of the pair have initialised their barriers before any remote arrival
  const uint32_t tmem_base = sh.tmem_base;
  const int total_tiles = sh.total_tiles;
  const int n_first = sh.first_tiles;
  const uint64_t limit = p.timeout_ns;
  const int rank = static_cast<int>(cluster_ctarank());
  const int cl_id = blockIdx.x / kPair, n_cl = gridDim.x / kPair;
  uint32_t mma_acc_uses = 0;   // MMA thread: tiles accumulated (accumulator buffer b: uses of b)
  // Tile t of the launch: whether it belongs to a1 (second) and its coordinates; each role
  // keeps its own expert cursors (c0 over a0's tiles, c1 over a1's).
  auto is_dgrad = [](bool second) { return !second && OP0 == kDgrad; };

  // ---------------------------------------------------------------- roles
  if (warp == 0) {
    // ===== TMA producer: packed ring, one unit (two k-blocks) per barrier =====
    if (lane == 0) {
      uint32_t uc = 0;
      ExpertCursor c0 = cursor_begin<OP0>(p), c1 = cursor_begin<kWgrad>(p1);
      uint32_t pend_mask = 0, pend_par = 0;
      for (int t = cl_id; t < total_tiles && !*abort_flag; t += n_cl) {
        bool second;
        const TileInfo ti = tile_at<OPS>(t, n_first, c0, c1, p, p1, rank, second);
        const bool dg = is_dgrad(second);
        const CUtensorMap* tm_p = second ? &tm_p1 : &tm_p0;
        const CUtensorMap* tm_s = second ? &tm_s1 : &tm_s0;
        const bool scale_tma = F::kFp4 && pick(second, p.scale_tma, p1.scale_tma) != 0;
        const uint32_t kb_bytes = F::kPBytes + (scale_tma ? F::kSBytes : 0);
        const int m0 = ti.mt * kTileM;
        const int pbatch = dg ? ti.e : 0;
        const int units = (ti.kblocks + kUnitKb - 1) / kUnitKb;
        bool ok = true;
        for (int j = 0; j < units; ++j, ++uc) {
          const Slot sl = ring_slot<F::kPUnits>(uc);
          if (!wait_phase(smem_u32(&sh.p_empty[sl.idx]), sl.par ^ 1u, abort_flag, p.err, limit)) { ok = false; break; }
          const uint32_t full = smem_u32(&sh.p_full[sl.idx]);
          const int nk = min(kUnitKb, ti.kblocks - kUnitKb * j);
          mbar_arrive_expect_tx(full, nk * kb_bytes);
          pend_mask |= 1u << sl.idx;
          pend_par = (pend_par & ~(1u << sl.idx)) | (sl.par << sl.idx);
          for (int h = 0; h < nk; ++h) {
            const int kb = kUnitKb * j + h;
            const int prow = dg ? kb * kTileK : ti.r0 + kb * kTileK;
            uint8_t* dst = ring_p + sl.idx * F::kPUnitBytes + h * F::kPStageBytes;
            if (FMT == BSQ_BF16) {
              tma_load_3d(smem_u32(dst), tm_p, full, m0, prow, pbatch);
              tma_load_3d(smem_u32(dst + kBoxBytes), tm_p, full, m0 + 64, prow, pbatch);
            } else {
              tma_load_3d(smem_u32(dst), tm_p, full, FMT == BSQ_FP8_E4M3_B128 ? m0 : m0 / 2, prow, pbatch);
              if (scale_tma) {
                // 16-byte aligned window holding this tile's scales (4 or 8 bytes per row)
                const int xs = (FMT == BSQ_MXFP4 ? (m0 >> 5) : (m0 >> 4)) & ~15;
                tma_load_3d(smem_u32(dst + F::kPBytes), tm_s, full, xs, prow, pbatch);
              }
            }
          }
        }
        if (!ok) break;
      }
      if (*abort_flag) drain_pending<F::kPUnits>(sh.p_full, pend_mask, pend_par, kDrainLimitNs);
    }
  } else if (warp == 3) {
    // ===== TMA producer: this CTA's half of the grad_out ring, one unit at a time =====
    if (lane == 0) {
      uint32_t uc = 0;
      ExpertCursor c0 = cursor_begin<OP0>(p), c1 = cursor_begin<kWgrad>(p1);
      uint32_t pend_mask = 0, pend_par = 0;
      for (int t = cl_id; t < total_tiles && !*abort_flag; t += n_cl) {
        bool second;
        const TileInfo ti = tile_at<OPS>(t, n_first, c0, c1, p, p1, rank, second);
        const bool dg = is_dgrad(second);
        const CUtensorMap* tm_g = second ? &tm_g1 : &tm_g0;
        const int b_mode = pick(second, p.b_mode, p1.b_mode);
        const int b_rows = pick(second, p.b_rows, p1.b_rows);
        const int half = rank * (mma_width(dg, ti.n_valid, b_mode) / 2);   // first n of this CTA's half
        // bytes of one k-block's half tile
        const uint32_t kb_bytes = b_mode == 1 ? b_rows * 128 : (b_mode == 2 ? b_rows : 2) * kBoxBytes;
        const int units = (ti.kblocks + kUnitKb - 1) / kUnitKb;
        bool ok = true;
        for (int j = 0; j < units; ++j, ++uc) {
          const Slot sl = ring_slot<kUStages>(uc);
          if (!wait_phase(smem_u32(&sh.op_empty[sl.idx]), sl.par ^ 1u, abort_flag, p.err, limit)) { ok = false; break; }
          const uint32_t full = smem_u32(&sh.b_full[sl.idx]);
          pend_mask |= 1u << sl.idx;
          pend_par = (pend_par & ~(1u << sl.idx)) | (sl.par << sl.idx);
          const int nk = min(kUnitKb, ti.kblocks - kUnitKb * j);
          mbar_arrive_expect_tx(full, nk * kb_bytes);
          for (int h = 0; h < nk; ++h) {
            const int kb = kUnitKb * j + h;
            const uint32_t dst = smem_u32(ring_b + sl.idx * kBUnitBytes + h * kBBytes);
            if (b_mode == 1) {
              // dgrad: b_rows tokens x 64 columns, K-major rows of 128 bytes
              tma_load_2d(dst, tm_g, full, kb * kTileK, ti.r0 + ti.nt * kTileN + half);
            } else if (b_mode == 2) {
              // wgrad: b_rows swizzle atoms x 64 tokens x 64 columns
              tma_load_3d(dst, tm_g, full, 0, ti.r0 + kb * kTileK, (ti.nt * kTileN + half) / 64);
            } else {
              // wgrad, N not a multiple of 64: two 64 x 64 boxes (the second may lie past N)
              for (int b = 0; b < 2; ++b)
                tma_load_2d(dst + b * kBoxBytes, tm_g, full, ti.nt * kTileN + half + 64 * b, ti.r0 + kb * kTileK);
            }
          }
        }
        if (!ok) break;
      }
      if (*abort_flag) drain_pending<kUStages>(sh.b_full, pend_mask, pend_par, kDrainLimitNs);
    }
  } else if (warp == 1) {
    // ===== MMA issuer: one thread of the even CTA drives the pair =====
    // This thread shares its scheduler with busy dequant warps, so its per-unit path is
    // kept short: one barrier wait, eight MMAs and one commit per unit of two k-blocks;
    // ring positions advance incrementally and the shared-memory descriptors are formed
    // by adding to the 14-bit start-address field (addresses < 256 KB).
    if (lane == 0 && rank == 0) {
      uint32_t iu = 0, pu = 0;   // ring slot and phase parity of the next unit
      ExpertCursor c0 = cursor_begin<OP0>(p), c1 = cursor_begin<kWgrad>(p1);
      uint32_t& acc = mma_acc_uses;
      const uint64_t adesc0 = sdesc_sw128(smem_u32(ring_a), kBoxBytes, 1024);    // A: MN-major, atoms of 64 m at 8 KB
      const uint64_t bdesc_k = sdesc_sw128(smem_u32(ring_b), 16, 1024);          // B (dgrad): K-major rows
      const uint64_t bdesc_mn = sdesc_sw128(smem_u32(ring_b), kBoxBytes, 1024);  // B (wgrad): MN-major
      const uint32_t a_full0 = smem_u32(&sh.a_full[0]), op_empty0 = smem_u32(&sh.op_empty[0]);
      // A unit is ready once both CTAs' relays have announced it: each has seen its CTA's A
      // rows written and its grad_out half landed.
      auto ready = [&](uint32_t s, uint32_t q) { return wait_phase<true>(a_full0 + 8 * s, q, abort_flag, p.err, limit); };
      // The units of one tile; BSTEP is the B descriptor step per 16 k (K-major: 32 bytes,
      // MN-major: one 2 KB row group).  Each unit's MMAs are queued, then the next unit is
      // awaited while they run, then the commit that frees the unit's slots (a commit takes
      // a slot of the tensor instruction queue; waiting after it would leave the pipe idle).
      // The next unit's slots were freed by a commit issued at least one unit earlier.
      auto run_tile = [&](auto bstep, uint64_t bdesc0, uint32_t d_tmem, uint32_t idesc, int kblocks) {
        constexpr uint32_t kBStep = decltype(bstep)::value;
        const int units = (kblocks + kUnitKb - 1) / kUnitKb;
        bool ok = ready(iu, pu);
        for (int j = 0; ok && j < units; ++j) {
          const int nk = min(kUnitKb, kblocks - kUnitKb * j);
          tc_fence_after();
          const uint64_t ad = adesc0 + iu * (kAUnitBytes >> 4);
          const uint64_t bd = bdesc0 + iu * (kBUnitBytes >> 4);
#pragma unroll
          for (int h = 0; h < kUnitKb; ++h) {
            if (h < nk) {
              umma_bf16_pair_k64<kBStep>(d_tmem, ad + h * (kABytes >> 4), bd + h * (kBBytes >> 4), idesc,
                                         (j | h) != 0 ? 1u : 0u);
            }
          }
          const uint32_t su = iu;
          if (++iu == kUStages) {
            iu = 0;
            pu ^= 1u;
          }
          if (j + 1 < units) ok = ready(iu, pu);
          umma_commit_pair(op_empty0 + 8 * su, kPairMask);
        }
        return ok;
      };
      for (int t = cl_id; t < total_tiles && !*abort_flag; t += n_cl) {
        bool second;
        const TileInfo ti = tile_at<OPS>(t, n_first, c0, c1, p, p1, rank, second);
        if (ti.kblocks == 0) continue;
        const bool dg = is_dgrad(second);
        const uint32_t buf = acc & 1u;
        const uint32_t acc_phase = (acc >> 1) & 1u;
        if (!wait_phase<true>(smem_u32(&sh.tmem_empty[buf]), acc_phase ^ 1u, abort_flag, p.err, limit)) break;
        tc_fence_after();
        const uint32_t n_mma = static_cast<uint32_t>(mma_width(dg, ti.n_valid, pick(second, p.b_mode, p1.b_mode)));
        const uint32_t idesc = idesc_bf16_f32(kPair * kTileM, n_mma, true, !dg);
        const uint32_t d_tmem = tmem_base + buf * kTileN;
        const bool ok = dg ? run_tile(std::integral_constant<uint32_t, (32 >> 4)>{}, bdesc_k, d_tmem, idesc, ti.kblocks)
                           : run_tile(std::integral_constant<uint32_t, (2048 >> 4)>{}, bdesc_mn, d_tmem, idesc, ti.kblocks);
        if (!ok) break;
        umma_commit_pair(smem_u32(&sh.tmem_full[buf]), kPairMask);
        ++acc;
      }
    }
  } else if (warp == 2) {
    // ===== operand-ready relay: one thread per CTA =====
    // Per unit: this CTA's dequant warps have written (and fenced) their A rows, and its
    // grad_out half has landed.  The even relay arrives on a_full expecting 4 bytes; the
    // odd relay's st.async delivers them with a cluster-scope release, because the even
    // CTA's MMA thread issues the MMA that reads the odd CTA's operands.
    if (lane == 0) {
      uint32_t uc = 0;
      ExpertCursor c0 = cursor_begin<OP0>(p), c1 = cursor_begin<kWgrad>(p1);
      const uint32_t a_full0 = smem_u32(&sh.a_full[0]);
      for (int t = cl_id; t < total_tiles && !*abort_flag; t += n_cl) {
        bool second;
        const TileInfo ti = tile_at<OPS>(t, n_first, c0, c1, p, p1, rank, second);
        const int units = (ti.kblocks + kUnitKb - 1) / kUnitKb;
        bool ok = true;
        for (int j = 0; j < units; ++j, ++uc) {
          const Slot sl = ring_slot<kUStages>(uc);
          if (!wait_phase(smem_u32(&sh.a_local[sl.idx]), sl.par, abort_flag, p.err, limit) ||
              !wait_phase(smem_u32(&sh.b_full[sl.idx]), sl.par, abort_flag, p.err, limit)) {
            ok = false;
            break;
          }
          if (rank == 0) {
            if (!p.drop_announce) mbar_arrive_expect_tx(a_full0 + 8 * sl.idx, 4);
          } else {
            st_async_tx_rank(smem_u32(&sh.sink), a_full0 + 8 * sl.idx, 0);
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp >= 4 && warp < 4 + R::kEpiWarps) {
    // ===== epilogue =====
    // Warp w reads TMEM lane quarter w % 4; the kEpiPerQuarter warps of a quarter take its
    // 16-column chunks in turn.
    const int q = warp & 3;                   // TMEM lane quarter
    const int sub = R::kEpiPerQuarter > 1 ? (warp - 4) >> 2 : 0;   // 0 .. kEpiPerQuarter-1
    const int i = q * 32 + lane;              // accumulator row = tile m index (permuted)
    const int mcol = lane_to_col<FMT>(i);
    const int lm = mcol - q * 32;             // column inside the warp's 32
    const uint32_t estage = smem_u32(ring_e) + (warp - 4) * F::kEpiStage;
    ExpertCursor c0 = cursor_begin<OP0>(p), c1 = cursor_begin<kWgrad>(p1);
    uint32_t acc = 0;
    for (int t = cl_id; t < total_tiles && !*abort_flag; t += n_cl) {
      bool second;
      const TileInfo ti = tile_at<OPS>(t, n_first, c0, c1, p, p1, rank, second);
      const int m = ti.mt * kTileM + mcol;
      const bool mok = m < p.Kc;
      __nv_bfloat16* obase = pick(second, p.out, p1.out);
      if (is_dgrad(second))
        obase += static_cast<int64_t>(ti.r0 + ti.nt * kTileN) * p.Kc + m;
      else
        obase += ti.e * pick(second, p.out_expert_stride, p1.out_expert_stride) +
                 static_cast<int64_t>(ti.nt * kTileN) * p.Kc + m;
      if (ti.kblocks == 0) {
        // wgrad of an expert without rows: exact zeros, 16 bytes per lane, 8 rows per warp store
        const int zc = ti.mt * kTileM + q * 32 + (lane & 3) * 8;
        __nv_bfloat16* zrow = pick(second, p.out, p1.out) + ti.e * pick(second, p.out_expert_stride, p1.out_expert_stride) +
                              static_cast<int64_t>(ti.nt * kTileN) * p.Kc + zc;
        if (zc < p.Kc)
          for (int n = (lane >> 2) + 8 * sub; n < ti.n_valid; n += 8 * R::kEpiPerQuarter)
            *reinterpret_cast<uint4*>(zrow + static_cast<int64_t>(n) * p.Kc) = make_uint4(0u, 0u, 0u, 0u);
        continue;
      }
      const uint32_t buf = acc & 1u;
      const uint32_t acc_phase = (acc >> 1) & 1u;
      ++acc;
      bool ok = wait_phase(smem_u32(&sh.tmem_full[buf]), acc_phase, abort_flag, p.err, limit);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int nchunks = (ti.n_valid + 15) >> 4;   // 16-column chunks of the accumulator
      // The even CTA's MMA thread reuses the accumulator once every epilogue warp of both
      // CTAs has released it: an even warp arrives expecting 4 bytes, an odd warp delivers
      // 4 bytes with an st.async (a cluster-scope release).
      auto release_acc = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0) mbar_arrive_expect_tx(smem_u32(&sh.tmem_empty[buf]), 4);
          else st_async_tx_rank(smem_u32(&sh.sink), smem_u32(&sh.tmem_empty[buf]), 0);
        }
      };
      if (sub >= nchunks) {
        release_acc();   // no chunk for this warp: release at once
        continue;
      }
      // The chunks of this warp: each TMEM load completes inside its own statement (see
      // tmem_ld_32x32b_x16_wait); the accumulator is released after the warp's last load.
      const uint32_t trow = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * kTileN;
      for (int c = sub; c < nchunks; c += R::kEpiPerQuarter) {
        uint32_t v[16];
        tmem_ld_32x32b_x16_wait(trow + c * 16, v);
        if (c + R::kEpiPerQuarter >= nchunks) release_acc();   // every TMEM read of this warp has completed
        uint32_t h[8];   // (n, n+1) pairs of this thread's column m, BF16
#pragma unroll
        for (int j = 0; j < 8; ++j) h[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
        if (F::kEpiStaged) {
          // [16 n][32 m] BF16 through this warp's staging area, then one TMA store (rows and
          // columns outside the output are clipped by the tensor map)
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            sts_u16(estage + j * 64 + lm * 2, (j & 1) ? (h[j >> 1] >> 16) : (h[j >> 1] & 0xFFFFu));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && ti.mt * kTileM + q * 32 < p.Kc) {
            tma_store_3d(&tm_o, estage, ti.mt * kTileM + q * 32, ti.nt * kTileN + c * 16, ti.e);
            bulk_commit();
          }
        } else if (mok) {
          const int nlim = min(16, ti.n_valid - c * 16);
          const int64_t step = p.Kc;
          unsigned short* o = reinterpret_cast<unsigned short*>(obase) + static_cast<int64_t>(c * 16) * step;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (j < nlim) *o = static_cast<unsigned short>((j & 1) ? (h[j >> 1] >> 16) : (h[j >> 1] & 0xFFFFu));
            o += step;
          }
        }
      }
    }
    if (F::kEpiStaged) {
      if (lane == 0) bulk_wait_all0();
      __syncwarp();
    }
  } else if (warp >= R::kFirstDeq) {
    // ===== dequantization =====
    // Thread -> (row r of the k-block, group g of 32 columns), plus rows r + kRowStep when
    // a thread decodes kRows rows.  A quarter-warp covers 4 consecutive rows x 2 groups,
    // so its 16-byte stores into the swizzled tile hit 8 distinct bank groups; each thread
    // needs one MX scale per row (two NVFP4, one FP8 block).
    const int dq = warp - R::kFirstDeq;
    const int team = dq / R::kDeqPerTeam;
    const int dw = dq % R::kDeqPerTeam;                        // warp within the team
    const int qtr = lane >> 3;
    const int r = dw * 8 + (qtr & 1) * 4 + (lane & 3);          // 0 .. kRowStep-1
    const int g = (qtr >> 1) * 2 + ((lane >> 2) & 1);           // 0..3
    // Shared addresses that do not change between k-blocks: the swizzled 16-byte store
    // slot of decoded group j (8 elements) of row r inside an A stage, and its packed
    // bytes inside a P stage (rows r + kRowStep: plus kRowStep rows; the swizzle phase
    // r & 7 is the same).  FP8 odd rows read their second 16 codes first (bank spread),
    // so their groups 0,1 hold chunks 2,3 of the row's 32 columns and vice versa.
    const uint32_t a_ring = smem_u32(ring_a), p_ring = smem_u32(ring_p);
    uint32_t st_off[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int chunk = (FMT == BSQ_FP8_E4M3_B128 && (r & 1)) ? (j ^ 2) : j;
      st_off[j] = (g >> 1) * kBoxBytes + r * 128 + ((((g & 1) * 4 + chunk) ^ (r & 7)) << 4);
    }
    const uint32_t p_off = F::kFp4 ? r * F::kPRowBytes + 16 * g : r * F::kPRowBytes + 32 * g + 16 * (r & 1);
    uint32_t uc = 0;   // units of earlier tiles: ring position of this tile's unit 0
    // One tile of the GEMM described by gp (a dgrad or a wgrad, fixed at compile time so
    // that the per-k-block work has no run-time op selection); false when the CTA aborted.
    auto deq_tile = [&](auto op_c, const TileInfo& ti, const Params& gp) -> bool {
      constexpr int OP = decltype(op_c)::value;
      const int m0 = ti.mt * kTileM;
      const int col0 = m0 + 32 * g;
      const bool col_ok = col0 < p.Kc;
      const int pbatch = OP == kDgrad ? ti.e : 0;
      float tscale = 0.f;
      if (FMT == BSQ_NVFP4) tscale = __ldg(gp.tensor_scale + pbatch);
      // this thread's scale byte(s) inside the staged 16-byte scale window of row r
      const uint32_t s_off = F::kPBytes + r * 16 + (FMT == BSQ_MXFP4 ? ((m0 >> 5) & 15) + g : ((m0 >> 4) & 15) + 2 * g);
      bool ok = true;
      const int units = (ti.kblocks + kUnitKb - 1) / kUnitKb;
      for (int j = 0; j < units; ++j) {
        // This team's k-block of the unit.  Past the tile's last k-block the team only
        // keeps the barrier counts: nothing is read or written and the MMA skips it.
        const int kb = kUnitKb * j + team;
        const bool present = kb < ti.kblocks;
        const Slot sa = ring_slot<kUStages>(uc + j);
        const Slot sp = ring_slot<F::kPUnits>(uc + j);
        const int prow0 = OP == kDgrad ? kb * kTileK : ti.r0 + kb * kTileK;
        const int kvalid = OP == kDgrad ? min(kTileK, p.N - kb * kTileK) : min(kTileK, ti.r1 - prow0);
        bool valid[R::kRows];
        // Scales that do not come through TMA are fetched before the wait.
        uint32_t sraw[R::kRows];
        float sf[R::kRows];
#pragma unroll
        for (int ps = 0; ps < R::kRows; ++ps) {
          const int rr = r + ps * R::kRowStep;
          valid[ps] = present && rr < kvalid && col_ok;
          sraw[ps] = 0;
          sf[ps] = 0.f;
          if (valid[ps]) {
            const int64_t grow = static_cast<int64_t>(pbatch) * gp.p_rows + prow0 + rr;
            if (FMT == BSQ_FP8_E4M3_B128)
              sf[ps] = __ldg(reinterpret_cast<const float*>(gp.scale) +
                             (static_cast<int64_t>(pbatch) * gp.scale_rblocks + ((prow0 + rr) >> gp.scale_shift)) *
                                 gp.scale_ld +
                             (col0 >> gp.scale_shift));
            else if (FMT == BSQ_MXFP4 && !gp.scale_tma)
              sraw[ps] = __ldg(gp.scale + grow * gp.scale_ld + (col0 >> 5));
            else if (FMT == BSQ_NVFP4 && !gp.scale_tma)
              sraw[ps] = static_cast<uint32_t>(__ldg(gp.scale + grow * gp.scale_ld + (col0 >> 4))) |
                         (static_cast<uint32_t>(__ldg(gp.scale + grow * gp.scale_ld + (col0 >> 4) + 1)) << 8);
          }
        }
        // Both teams wait on every phase of the packed slot (in unit order) and both count
        // out of it, present or not.
        ok = wait_phase(smem_u32(&sh.p_full[sp.idx]), sp.par, abort_flag, p.err, limit);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        // ---- read this thread's packed bytes (and scales) out of the packed ring
        const uint32_t pst = p_ring + sp.idx * F::kPUnitBytes + team * F::kPStageBytes;
        uint4 wa[R::kRows], wb[R::kRows];
        uint32_t v[4][4];   // 4 groups of 8 elements, 4 BF16 pairs each (permuted inside the group)
#pragma unroll
        for (int ps = 0; ps < R::kRows; ++ps) {
          wa[ps] = make_uint4(0, 0, 0, 0);
          wb[ps] = make_uint4(0, 0, 0, 0);
          const uint32_t po = p_off + ps * R::kRowStep * F::kPRowBytes;
          if (FMT != BSQ_BF16 && valid[ps]) {
            if (F::kFp4) {
              if (gp.scale_tma) {
                const uint32_t so = s_off + ps * R::kRowStep * 16;
                sraw[ps] = FMT == BSQ_MXFP4 ? lds_u8(pst + so) : lds_u16(pst + so);
              }
              wa[ps] = lds128(pst + po);
            } else {
              // rows 128 bytes apart share banks: odd rows read their second half first
              // (the store slots above put the groups back in place)
              wa[ps] = lds128(pst + po);
              wb[ps] = lds128(pst + (po ^ 16u));
            }
          }
        }
        if (FMT == BSQ_BF16 && present) {
          // BF16 operand: the TMA tile is already in the swizzled layout; copy this
          // thread's four 16-byte chunks (zero outside the contraction).
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const uint4 c = r < kvalid ? lds128(pst + st_off[jj]) : make_uint4(0, 0, 0, 0);
            v[jj][0] = c.x; v[jj][1] = c.y; v[jj][2] = c.z; v[jj][3] = c.w;
          }
        }
        // The producer refills this slot by TMA (the async proxy) once every dequant warp has
        // arrived; this lane's plain loads from it must be performed first.  Without the fence
        // nothing orders them, and a load still queued behind other shared-memory traffic of
        // the SM can read the next unit's bytes.
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.p_empty[sp.idx]));   // this warp is done with the packed slot
        // ---- decode the first row into registers while the operand slot may still be busy
        if (FMT != BSQ_BF16 && present) decode_row<FMT>(wa[0], wb[0], sraw[0], sf[0], tscale, valid[0], v);
        // The unit's operand and grad_out slots are free once its previous MMAs completed.
        ok = wait_phase(smem_u32(&sh.op_empty[sa.idx]), sa.par ^ 1u, abort_flag, p.err, limit);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if (present) {
          // group jj of this thread = 8-element chunk 4g + jj of the row: swizzle column
          // g/2, 16-byte slot (4(g&1) + jj) XOR (r & 7)
          const uint32_t ast = a_ring + sa.idx * kAUnitBytes + team * kABytes;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) sts128(ast + st_off[jj], v[jj][0], v[jj][1], v[jj][2], v[jj][3]);
#pragma unroll
          for (int ps = 1; ps < R::kRows; ++ps) {
            decode_row<FMT>(wa[ps], wb[ps], sraw[ps], sf[ps], tscale, valid[ps], v);
            const uint32_t ar = ast + ps * R::kRowStep * 128;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) sts128(ar + st_off[jj], v[jj][0], v[jj][1], v[jj][2], v[jj][3]);
          }
          if (OP == kWgrad && kvalid < kTileK) {
            // grad_out rows past the expert (possibly uninitialised past offsets[E-1]) must
            // not reach the products: once this CTA's grad_out half has landed, zero them in
            // both boxes of the half.
            ok = wait_phase(smem_u32(&sh.b_full[sa.idx]), sa.par, abort_flag, p.err, limit);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const uint32_t b_tile = smem_u32(ring_b + sa.idx * kBUnitBytes + team * kBBytes);
            const int dt = dw * 32 + lane;
            for (int idx = dt; idx < (kTileK - kvalid) * 8 * 2; idx += 32 * R::kDeqPerTeam) {
              const int box = idx / ((kTileK - kvalid) * 8);
              const int rem = idx % ((kTileK - kvalid) * 8);
              const int rr = kvalid + rem / 8, c = rem % 8;
              sts128(b_tile + box * kBoxBytes + rr * 128 + c * 16, 0u, 0u, 0u, 0u);
            }
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.a_local[sa.idx]));   // this CTA's relay passes it on
      }
      uc += units;
      return ok;
    };
    // The first GEMM's tiles, then (kBoth) the second's: two loops, so that only one expert
    // cursor is live at a time.
    int t = cl_id;
    bool ok = true;
    {
      ExpertCursor c0 = cursor_begin<OP0>(p);
      const int end0 = OPS == kBoth ? n_first : total_tiles;
      for (; ok && t < end0 && !*abort_flag; t += n_cl)
        ok = deq_tile(std::integral_constant<int, OP0>{}, decode_tile<OP0>(t, c0, p, rank), p);
    }
    if (OPS == kBoth) {
      ExpertCursor c1 = cursor_begin<kWgrad>(p1);
      for (; ok && t < total_tiles && !*abort_flag; t += n_cl)
        ok = deq_tile(std::integral_constant<int, kWgrad>{}, decode_tile<kWgrad>(t - n_first, c1, p1, rank), p1);
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (warp == 1 && lane == 0 && rank == 0) {
    // Every MMA this thread issued has completed (and read the odd CTA's shared memory)
    // once the drain barrier fires.
    umma_commit_pair(smem_u32(&sh.drain), 1);
    uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(smem_u32(&sh.drain), 0) && global_timer_ns() - t0 < kDrainLimitNs) {
    }
    // The odd CTA's st.async releases of the last accumulators are never waited on by the
    // main loop; they must land before this CTA's shared memory goes away.
    if (!*abort_flag) {
      for (uint32_t b = 0; b < 2; ++b) {
        const uint32_t uses = (mma_acc_uses + 1u - b) / 2u;
        if (uses == 0) continue;
        t0 = global_timer_ns();
        while (!mbar_try_wait(smem_u32(&sh.tmem_empty[b]), (uses - 1u) & 1u) &&
               global_timer_ns() - t0 < kDrainLimitNs) {
        }
      }
    }
  }
  if (rank == 0 && *abort_flag) {
    // After an abort the odd CTA may still have st.async announcements in flight to this
    // CTA, which nothing waits for: give them time to land before the shared memory goes.
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < kAbortSettleNs) {
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // No CTA leaves while its peer may still arrive on its barriers or read its operands.
  cluster_sync();
  if (warp == 2) tmem_dealloc_pair(tmem_base, kTmemCols);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

}  // namespace

// Tiled tensor map through the driver entry point (no link against libcuda); also used by
// the small-M kernel.
bool encode_map(CUtensorMap* m, CUtensorMapDataType dt, uint32_t rank, const void* base, const uint64_t* dims,
                const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle sw) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  const uint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, dt, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

// Tensor maps and parameters of one GEMM; *bound is an upper bound of its pair tiles (the
// exact count depends on the offsets, which only the device reads).
template <int FMT>
int prepare_op(const GemmArgs& a, OpArgs& o, int64_t* bound, const char** msg) {
  const bool dgrad = a.op == kDgrad;
  int b_mode = 0, b_rows = 0;
  {
    // this CTA's half of a k-block's grad_out tile in a single TMA copy where the shape allows it
    const uint64_t dims[2] = {static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.S)};
    const uint64_t strides[1] = {static_cast<uint64_t>(a.N) * 2};
    bool ok = false;
    if (dgrad) {
      b_rows = static_cast<int>(a.S < kBHalf ? a.S : kBHalf);
      const uint32_t box[2] = {64, static_cast<uint32_t>(b_rows)};
      ok = encode_map(&o.tm_g, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.g, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
      b_mode = 1;
    } else if (a.N % 64 == 0) {
      // [N/64 swizzle columns][S tokens][64 columns] view of grad_out
      b_rows = static_cast<int>(a.N / 64 < kBHalf / 64 ? a.N / 64 : kBHalf / 64);
      const uint64_t d3[3] = {64, static_cast<uint64_t>(a.S), static_cast<uint64_t>(a.N / 64)};
      const uint64_t s3[2] = {static_cast<uint64_t>(a.N) * 2, 128};
      const uint32_t box[3] = {64, 64, static_cast<uint32_t>(b_rows)};
      ok = encode_map(&o.tm_g, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.g, d3, s3, box, CU_TENSOR_MAP_SWIZZLE_128B);
      b_mode = 2;
    }
    if (!ok && !dgrad) {
      const uint32_t box[2] = {64, 64};
      ok = encode_map(&o.tm_g, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.g, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
      b_mode = 0;
    }
    if (!ok) {
      *msg = "tensor map encoding failed for grad_out";
      return -1;
    }
  }
  {
    uint64_t row_bytes;
    CUtensorMapDataType dt;
    uint32_t box0;
    CUtensorMapSwizzle sw;
    uint64_t inner;
    if (FMT == BSQ_BF16) {
      dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16; inner = a.kc; row_bytes = a.kc * 2; box0 = 64; sw = CU_TENSOR_MAP_SWIZZLE_128B;
    } else if (FMT == BSQ_FP8_E4M3_B128) {
      dt = CU_TENSOR_MAP_DATA_TYPE_UINT8; inner = a.kc; row_bytes = a.kc; box0 = kTileM; sw = CU_TENSOR_MAP_SWIZZLE_NONE;
    } else {
      dt = CU_TENSOR_MAP_DATA_TYPE_UINT8; inner = a.kc / 2; row_bytes = a.kc / 2; box0 = kTileM / 2; sw = CU_TENSOR_MAP_SWIZZLE_NONE;
    }
    const uint64_t dims[3] = {inner, static_cast<uint64_t>(a.p_rows), static_cast<uint64_t>(a.p_batch)};
    const uint64_t strides[2] = {row_bytes, row_bytes * static_cast<uint64_t>(a.p_rows)};
    const uint32_t box[3] = {box0, static_cast<uint32_t>(kTileK), 1};
    if (!encode_map(&o.tm_p, dt, 3, a.p_data, dims, strides, box, sw)) {
      *msg = "tensor map encoding failed for the packed operand";
      return -1;
    }
  }
  // wgrad output [E][N][Kc] as TMA store boxes of 16 rows x 32 columns
  o.tm_o = o.tm_p;
  if (!dgrad) {
    const uint64_t dims[3] = {static_cast<uint64_t>(a.kc), static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.E)};
    const uint64_t strides[2] = {static_cast<uint64_t>(a.kc) * 2, static_cast<uint64_t>(a.kc * a.N) * 2};
    const uint32_t box[3] = {32, 16, 1};
    if (!encode_map(&o.tm_o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.out, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE)) {
      *msg = "tensor map encoding failed for the output";
      return -1;
    }
  }
  // FP4 scale tiles through TMA when the scale row pitch is a multiple of 16 bytes.
  o.tm_s = o.tm_p;
  int scale_tma = 0;
  if (FMT == BSQ_MXFP4 || FMT == BSQ_NVFP4) {
    const uint64_t srow = FMT == BSQ_MXFP4 ? a.kc / 32 : a.kc / 16;
    if (srow % 16 == 0 && (reinterpret_cast<uintptr_t>(a.p_scale) & 15u) == 0) {
      const uint64_t dims[3] = {srow, static_cast<uint64_t>(a.p_rows), static_cast<uint64_t>(a.p_batch)};
      const uint64_t strides[2] = {srow, srow * static_cast<uint64_t>(a.p_rows)};
      const uint32_t box[3] = {16, static_cast<uint32_t>(kTileK), 1};
      if (!encode_map(&o.tm_s, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a.p_scale, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_NONE)) {
        *msg = "tensor map encoding failed for the scales";
        return -1;
      }
      scale_tma = 1;
    }
  }
  Params& p = o.p;
  p.scale_tma = scale_tma;
  p.b_mode = b_mode;
  p.b_rows = b_rows;
  p.scale = static_cast<const uint8_t*>(a.p_scale);
  p.tensor_scale = a.p_tensor_scale;
  p.offsets = a.offsets;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.err = a.err;
  p.out_expert_stride = dgrad ? 0 : a.N * a.kc;
  p.p_rows = a.p_rows;
  p.E = static_cast<int32_t>(a.E);
  p.S = static_cast<int32_t>(a.S);
  p.N = static_cast<int32_t>(a.N);
  p.Kc = static_cast<int32_t>(a.kc);
  p.num_m = static_cast<int32_t>((a.kc + kTileM - 1) / kTileM);
  p.num_mg = (p.num_m + kPair - 1) / kPair;
  const bool per_tensor = a.fmt == BSQ_FP8_E4M3_TENSOR;
  p.scale_ld = FMT == BSQ_MXFP4 ? static_cast<int32_t>(a.kc / 32)
               : FMT == BSQ_NVFP4 ? static_cast<int32_t>(a.kc / 16)
               : per_tensor       ? 1
                                  : static_cast<int32_t>((a.kc + 127) / 128);
  p.scale_rblocks = per_tensor ? 1 : static_cast<int32_t>((a.p_rows + 127) / 128);
  p.scale_shift = fp8_scale_shift(a.fmt);
  p.timeout_ns = wait_limit_ns();
  // Test hook (failure detection without a GPU fault): with BSQ_TEST_DROP_ANNOUNCE=1 the
  // MMA thread's first operand-ready wait can never complete, so it runs out of time and
  // the kernel takes its orderly abort.
  const char* drop = std::getenv("BSQ_TEST_DROP_ANNOUNCE");
  p.drop_announce = drop && drop[0] == '1' ? 1 : 0;
  p.tail_rows = dgrad && a.offsets ? a.tail_rows : 0;
  const int64_t nn = (a.N + kTileN - 1) / kTileN;
  *bound = dgrad ? p.num_mg * ((a.S + kTileN - 1) / kTileN + a.E) : p.num_mg * nn * a.E;
  return 0;
}

// Launch one GEMM (OPS = its op; ops[0]) or a dgrad and a wgrad over the same grad_out
// (OPS = kBoth; ops[0] the dgrad, ops[1] the wgrad).
template <int FMT, int OPS>
int launch_typed(const GemmArgs* ops, const char** msg) {
  OpArgs a0, a1;
  int64_t b0 = 0, b1 = 0;
  if (prepare_op<FMT>(ops[0], a0, &b0, msg) != 0) return -1;
  if (OPS == kBoth) {
    if (prepare_op<FMT>(ops[1], a1, &b1, msg) != 0) return -1;
  } else {
    a1 = a0;
  }
  const int64_t bound = b0 + b1;
  const GemmArgs& a = ops[0];
  static_assert(Fmt<FMT>::kRingBytes + sizeof(SharedTail) + 1024 <= 232448, "rings exceed the 227 KB of shared memory per CTA");
  static_assert(Fmt<FMT, true>::kRingBytes + sizeof(SharedTail) + 1024 <= 232448, "rings exceed the 227 KB of shared memory per CTA");
  size_t smem = static_cast<size_t>(Fmt<FMT>::kRingBytes) + sizeof(SharedTail) + 1024;
  // Kernel: wgrad of a packed format whose groups average fewer than 1024 rows (a tile of
  // at most 16 k-blocks, where the epilogue sets the pace) takes the short-tile variant
  // (more epilogue warps).  BSQ_GEMM_SHORT_TILES=1 / 0 forces one or the other.
  auto kern = bsq_gemm_kernel<FMT, OPS, false>;
  bool short_tiles = false;
  if constexpr (OPS == kWgrad && FMT != BSQ_BF16) {
    const char* env = std::getenv("BSQ_GEMM_SHORT_TILES");
    if (env && (env[0] == '0' || env[0] == '1')) short_tiles = env[0] == '1';
    else short_tiles = a.S < 1024 * a.E;
    if (short_tiles) {
      kern = bsq_gemm_kernel<FMT, OPS, true>;
      smem = static_cast<size_t>(Fmt<FMT, true>::kRingBytes) + sizeof(SharedTail) + 1024;
    }
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPair;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // Persistent grid: as many pairs as can be resident at once (a GPC with an odd number of
  // free SMs leaves one idle), never more than there are pair tiles.  The count is kept per
  // kernel variant and device.
  static std::atomic<int> max_clusters_of[2][kMaxDevices];
  int dev = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess && (dev < 0 || dev >= kMaxDevices)) e = cudaErrorInvalidDevice;
  int max_clusters = e == cudaSuccess ? max_clusters_of[short_tiles][dev].load() : 0;
  if (e == cudaSuccess && max_clusters == 0) {
    cfg.gridDim = dim3(kPair * (a.num_sms / kPair));
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    max_clusters = n > 0 ? n : a.num_sms / kPair;
    max_clusters_of[short_tiles][dev].store(max_clusters);
  }
  int64_t clusters = bound < max_clusters ? bound : max_clusters;
  if (clusters < 1) clusters = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * kPair));
  if (e == cudaSuccess)
    e = cudaLaunchKernelEx(&cfg, kern, a0.tm_p, a0.tm_g, a0.tm_s, a1.tm_p, a1.tm_g, a1.tm_s, a0.tm_o, a0.p, a1.p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    *msg = cudaGetErrorString(e);
    return static_cast<int>(e);
  }
  return 0;
}

}  // namespace

int launch_gemm(const GemmArgs& a, const char** msg) {
  const int kf = kernel_fmt(a.fmt);
#define BSQ_CASE(F_, O_) \
  if (kf == F_ && a.op == O_) return launch_typed<F_, O_>(&a, msg);
  BSQ_CASE(BSQ_BF16, kDgrad)
  BSQ_CASE(BSQ_BF16, kWgrad)
  BSQ_CASE(BSQ_FP8_E4M3_B128, kDgrad)
  BSQ_CASE(BSQ_FP8_E4M3_B128, kWgrad)
  BSQ_CASE(BSQ_MXFP4, kDgrad)
  BSQ_CASE(BSQ_MXFP4, kWgrad)
  BSQ_CASE(BSQ_NVFP4, kDgrad)
  BSQ_CASE(BSQ_NVFP4, kWgrad)
#undef BSQ_CASE
  *msg = "unsupported format/op";
  return -1;
}

int launch_gemm_backward(const GemmArgs& dgrad, const GemmArgs& wgrad, const char** msg) {
  if (dgrad.op != kDgrad || wgrad.op != kWgrad || kernel_fmt(dgrad.fmt) != kernel_fmt(wgrad.fmt) || dgrad.E != wgrad.E ||
      dgrad.S != wgrad.S || dgrad.N != wgrad.N || dgrad.kc != wgrad.kc || dgrad.g != wgrad.g ||
      dgrad.offsets != wgrad.offsets) {
    *msg = "a fused backward needs one grad_out, one packed format, one K and one set of offsets";
    return -1;
  }
  const GemmArgs ops[2] = {dgrad, wgrad};
  switch (kernel_fmt(dgrad.fmt)) {
    case BSQ_BF16: return launch_typed<BSQ_BF16, kBoth>(ops, msg);
    case BSQ_FP8_E4M3_B128: return launch_typed<BSQ_FP8_E4M3_B128, kBoth>(ops, msg);
    case BSQ_MXFP4: return launch_typed<BSQ_MXFP4, kBoth>(ops, msg);
    case BSQ_NVFP4: return launch_typed<BSQ_NVFP4, kBoth>(ops, msg);
    default: break;
  }
  *msg = "unsupported format";
  return -1;
}

}  // namespace bsq
