// Pieces shared by the prefill kernels: the per-translation-unit device status
// word and the bounded waits every role of a prefill CTA uses.
#pragma once

#include <math_constants.h>

#include "checked.cuh"
#include "common.cuh"
#include "ptx.cuh"
#include "schedule.cuh"

namespace attn {

static __device__ unsigned int g_prefill_status;

// The polling loop of the bounded waits below, after a first failed poll.
__device__ __forceinline__ bool pf_spin(uint32_t a, uint32_t parity, volatile uint32_t* abort, uint32_t site) {
  uint64_t t0 = 0;
#pragma unroll 1
  for (uint32_t it = 0;; ++it) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(a, parity)) return true;
    if (*abort) return false;
    if ((it & 15u) == 15u) {
      const uint64_t now = global_timer_ns();
      if (t0 == 0) t0 = now;
      const bool late = now - t0 > kWaitTimeoutNs;
      if (late) atomicOr(&g_prefill_status, kStatusTimeout | (site << kStatusSiteShift));
      if (late || (*reinterpret_cast<volatile unsigned int*>(&g_prefill_status) & kStatusTimeout)) {
        *abort = 1u;
        return false;
      }
    }
  }
}

// Out-of-line rest of a bounded wait (one copy per translation unit).
static __device__ __noinline__ bool pf_wait_slow(uint32_t a, uint32_t parity, volatile uint32_t* abort,
                                                 uint32_t site) {
  return pf_spin(a, parity, abort, site);
}
// Bounded wait used by every role; also gives up once another CTA of any
// launch has reported a timeout, so a broken pipeline ends quickly.  The
// barrier is polled first: the clock and the device-wide status word (a
// global-memory round trip) are read only every 512 failed polls, because
// these waits sit on the critical path between the MMA and softmax roles.
// The first 32 polls are inline and the rest of the wait is a call: the call
// site stays small (the kernels are sensitive to instruction-cache pressure)
// while the call, and the registers it saves, stay off the common path where
// a wait ends within a few polls.  This measured 1-3 % faster than a fully
// inline wait in the paired kernel, where calling out after the first failed
// poll instead raised spills at its register limit and cost 6 %.
__device__ __forceinline__ bool pf_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort, uint32_t site) {
  const uint32_t a = smem_u32(bar);
#pragma unroll 1
  for (int i = 0; i < 32; ++i)
    if (mbar_try_wait(a, parity)) return true;
  return pf_wait_slow(a, parity, abort, site);
}

// The same wait with a single inline poll before the call: the head-dim-256
// kernel, with registers to spare, measured 4 % faster with it than with a
// fully inline wait.
__device__ __forceinline__ bool pf_wait_outlined(uint64_t* bar, uint32_t parity, volatile uint32_t* abort,
                                                 uint32_t site) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  return pf_wait_slow(a, parity, abort, site);
}

// Visible keys of a 32-key chunk whose first key is key c0 of its tile: bit i
// is set iff flo <= c0 + i < lim.  The limits come clamped to [0, tile keys],
// so a masked tile's scores are tested with 32-bit masks, not one pair of
// 64-bit compares per score.
__device__ __forceinline__ uint32_t chunk_mask(int c0, int flo, int lim) {
  const int lo = min(max(flo - c0, 0), 32), hi = min(max(lim - c0, 0), 32);
  const uint32_t below_hi = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
  const uint32_t below_lo = lo >= 32 ? 0xffffffffu : ((1u << lo) - 1u);
  return below_hi & ~below_lo;
}

// Scores of a 32-key chunk outside `mask` become -inf.
__device__ __forceinline__ void apply_mask(uint32_t (&r)[32], uint32_t mask, uint32_t ninf) {
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = ((mask >> i) & 1u) ? r[i] : ninf;
}

// Clamp a key limit of a tile of `keys` keys to [0, keys].
__device__ __forceinline__ int clamp_limit(long long v, int keys) {
  return (int)(v < 0 ? 0 : (v > keys ? keys : v));
}

// Wait used only while tearing down after an abort: ignores the abort flag.
__device__ __forceinline__ bool pf_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (global_timer_ns() - t0 > kWaitTimeoutNs) {
      atomicOr(&g_prefill_status, kStatusTimeout | (0x80u << kStatusSiteShift));
      return false;
    }
  }
  return true;
}

inline unsigned int prefill_take_status_impl(cudaStream_t s) {
  if (cudaStreamSynchronize(s) != cudaSuccess) return kStatusTimeout;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_prefill_status, sizeof(v)) != cudaSuccess) return kStatusTimeout;
  if (v != 0) {
    const unsigned int zero = 0;
    cudaMemcpyToSymbol(g_prefill_status, &zero, sizeof(zero));
  }
  return v;
}

}  // namespace attn
