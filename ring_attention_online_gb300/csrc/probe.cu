// Tensor-pipe rate probe: one CTA issues back-to-back tcgen05.mma kind::f16
// M=128 N=128 K=16 MMAs from one thread (bf16 operands in shared memory, fp32
// accumulator in TMEM) and times them with the SM clock.  It gives the per-SM
// dense bf16 rate from which the nominal roofline denominator is built.
#include "common.cuh"
#include "ptx.cuh"

namespace attn {

static __device__ unsigned int g_probe_status;

__global__ void __launch_bounds__(128, 1) probe_mma_kernel(int groups, unsigned long long* out) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t done;
  __shared__ uint32_t tslot, abort_flag;
  // A and B: one 128-row x 64-column bf16 block each (16 KB, 128-byte swizzle), zeros
  for (int i = threadIdx.x; i < 32768 / 16; i += blockDim.x) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&done, 1);
    fence_barrier_init();
  }
  if (threadIdx.x < 32) {
    tmem_alloc(&tslot, 128);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tm = tslot;
  if (threadIdx.x == 0) {
    constexpr uint32_t idesc = idesc_f16_f32acc(128, 128, true, false);
    const uint32_t a = smem_u32(sm);
    const uint64_t ad = smem_desc_sw128(a, 16, 1024), bd = smem_desc_sw128(a + 16384, 16, 1024);
    const long long t0 = clock64();
#pragma unroll 1
    for (int g = 0; g < groups; ++g) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)  // K = 16 per MMA: 32 bytes of each 128-byte row, twice over the block
        mma_ss(tm, desc_advance(ad, (ks & 3) * 32), desc_advance(bd, (ks & 3) * 32), idesc, (g | ks) != 0);
    }
    mma_commit(&done);
    // the issuing thread's wait returns once its MMAs have all completed
    const bool ok = mbar_wait_bounded(&done, 0, &abort_flag, &g_probe_status, kStatusTimeout, kWaitTimeoutNs);
    const long long t1 = clock64();
    out[0] = static_cast<unsigned long long>(t1 - t0);
    out[1] = ok ? 0ull : 1ull;
  }
  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after_sync();
    tmem_dealloc(tm, 128);
  }
}

attn_status_t launch_probe_mma(unsigned long long* out, int groups, cudaStream_t s) {
  probe_mma_kernel<<<1, 128, 32768 + 1024, s>>>(groups, out);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn
