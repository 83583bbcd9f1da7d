// Prefill kernels for head dimension 256 (fp16 / bf16; dense, partial, jagged,
// window): CTA pairs with tcgen05 cta_group::2 (prefill_cta2_kernel.cuh).
#include "prefill_cta2_kernel.cuh"

namespace attn {

attn_status_t launch_prefill_d256(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                 const CUtensorMap& mv, int mode, bool bf16, dim3 grid, cudaStream_t s) {
  return launch_cta2_dispatch<256>(p, mq, mk, mv, mode, bf16, grid, s);
}

unsigned int prefill_d256_take_status(cudaStream_t s) { return prefill_take_status_impl(s); }

}  // namespace attn
