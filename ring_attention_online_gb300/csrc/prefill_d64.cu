// Prefill kernels for head dimension 64 (fp16 / bf16; dense, partial, jagged).
#include "prefill_kernel.cuh"

namespace attn {

attn_status_t launch_prefill_d64(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                 const CUtensorMap& mv, int mode, bool bf16, dim3 grid, cudaStream_t s) {
  return launch_prefill_dispatch<64>(p, mq, mk, mv, mode, bf16, grid, s);
}

unsigned int prefill_d64_take_status(cudaStream_t s) { return prefill_take_status_impl(s); }

}  // namespace attn
