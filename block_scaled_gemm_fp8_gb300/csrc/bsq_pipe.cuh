// bsq_pipe.cuh -- pipeline pieces the persistent pair-MMA kernels share: bounded mbarrier
// waits that stop the CTA pair instead of hanging, ring positions, and the drain of an
// aborting producer's copies.
#pragma once

#include <cstdint>

#include "bsq_ptx.cuh"
#include "../../include/bsq.h"

namespace bsq {

__device__ __forceinline__ void record_error(int32_t* err, int32_t code) { atomicCAS(err, 0, code); }

// Bounded wait on an mbarrier phase; false when the CTA aborted or the limit ran out.  A
// timeout stops this CTA and its peer (both abort flags sit at the same shared offset).
// CL: the barrier receives arrivals from the peer CTA (acquire at cluster scope).
template <bool CL>
__device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                             int32_t* err, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (CL ? mbar_try_wait_sleep_cl(bar, parity, 20000u) : mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1u;
      st_rank_u32(smem_u32(const_cast<uint32_t*>(abort_flag)), cluster_ctarank() ^ 1u, 1u);
      record_error(err, BSQ_DEVERR_TIMEOUT);
      return false;
    }
  }
}
template <bool CL = false>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                           int32_t* err, uint64_t limit_ns) {
  if (CL ? mbar_try_wait_cl(bar, parity) : mbar_try_wait(bar, parity)) return true;
  return wait_phase_slow<CL>(bar, parity, abort_flag, err, limit_ns);
}

// Ring position of the u-th unit: slot and the parity of the phase it fills.
struct Slot {
  int idx;
  uint32_t par;
};
template <int N>
__device__ __forceinline__ Slot ring_slot(uint32_t u) {
  return Slot{static_cast<int>(u % N), (u / N) & 1u};
}

// Let the TMA copies this thread issued into the given slots land (orderly abort).
template <int N>
__device__ __forceinline__ void drain_pending(uint64_t* full, uint32_t mask, uint32_t par, uint64_t limit) {
  for (int s = 0; s < N; ++s)
    if (mask & (1u << s)) {
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(smem_u32(&full[s]), (par >> s) & 1u) && global_timer_ns() - t0 < limit) {
      }
    }
}


}  // namespace bsq
