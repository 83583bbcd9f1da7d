// Prefill kernels for head dimension 64 (fp16 / bf16; dense, partial, jagged):
// two 128-row Q sub-tiles per CTA sharing each K/V tile.
#include "prefill_pair_kernel.cuh"

namespace attn {

attn_status_t launch_prefill_d64(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                 const CUtensorMap& mv, int mode, bool bf16, dim3 grid, cudaStream_t s) {
  return launch_pair_dispatch<64>(p, mq, mk, mv, mode, bf16, grid, s);
}

unsigned int prefill_d64_take_status(cudaStream_t s) { return prefill_take_status_impl(s); }

}  // namespace attn
