// Pieces shared by the prefill kernels: the per-translation-unit device status
// word and the bounded waits every role of a prefill CTA uses.
#pragma once

#include <math_constants.h>

#include "common.cuh"
#include "ptx.cuh"
#include "schedule.cuh"

namespace attn {

static __device__ unsigned int g_prefill_status;

// Bounded wait used by every role; also gives up as soon as another CTA of
// any launch has reported a timeout (so a broken pipeline ends quickly).
__device__ __forceinline__ bool pf_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort, uint32_t site) {
  if (mbar_try_wait(smem_u32(bar), parity)) return true;
  if (*reinterpret_cast<volatile unsigned int*>(&g_prefill_status) & kStatusTimeout) {
    *abort = 1u;
    return false;
  }
  return mbar_wait_bounded(bar, parity, abort, &g_prefill_status, kStatusTimeout | (site << kStatusSiteShift),
                           kWaitTimeoutNs);
}

// Wait used only while tearing down after an abort: ignores the abort flag.
__device__ __forceinline__ void pf_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (global_timer_ns() - t0 > kWaitTimeoutNs) {
      atomicOr(&g_prefill_status, kStatusTimeout | (0x80u << kStatusSiteShift));
      return;
    }
  }
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
