// Prefill kernels for head dimension 256 (fp16 / bf16; dense, partial, jagged).
#include "prefill_kernel.cuh"

namespace attn {

attn_status_t launch_prefill_d256(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                 const CUtensorMap& mv, int mode, bool bf16, dim3 grid, cudaStream_t s) {
  return launch_prefill_dispatch<256>(p, mq, mk, mv, mode, bf16, grid, s);
}

unsigned int prefill_d256_take_status(cudaStream_t s) { return prefill_take_status_impl(s); }

}  // namespace attn
