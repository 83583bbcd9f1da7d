// Fold of C partial triplets per row, then the final normalisation (the fold
// itself, and its sources, are in merge.cuh).
//
// One warp per output row.  HBM-bound.
#include "merge.cuh"

namespace attn {

static __device__ unsigned int g_merge_status;  // checked builds: store bounds

template <int D, bool kBf16>
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ m, const float* __restrict__ l,
                                                    const float* __restrict__ o, int C, int B, int S_q, int H,
                                                    void* __restrict__ out, float* __restrict__ lse) {
  const long long rows = (long long)B * S_q * H;
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  // output row order (b, s, h) follows O's layout [B, S_q, H, D]; m, l and
  // LSE are [.., B, H, S_q]
  const int h = (int)(row % H);
  const long long bs = row / H;
  const int s = (int)(bs % S_q);
  const long long b = bs / S_q;
  const size_t ml_idx = ((size_t)b * H + h) * S_q + s;
  merge_row<D, kBf16>(m, l, o, C, (size_t)B * H * S_q, ml_idx, (size_t)rows * D, (size_t)row * D, out, lse, ml_idx,
                      lane, rows, &g_merge_status);
}

template <int D, bool kBf16>
static attn_status_t launch_merge_t(const float* m, const float* l, const float* o, int C, int B, int S_q, int H,
                                    void* out, float* lse, cudaStream_t s) {
  const long long rows = (long long)B * S_q * H;
  const long long blocks = (rows + 7) / 8;
  if (blocks == 0) return ATTN_OK;
  if (blocks > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  merge_kernel<D, kBf16><<<(unsigned)blocks, 256, 0, s>>>(m, l, o, C, B, S_q, H, out, lse);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t launch_merge(const float* m, const float* l, const float* o, int C, int B, int S_q, int H, int D,
                           void* out, bool out_bf16, float* lse, cudaStream_t s) {
  switch (D) {
    case 64: return out_bf16 ? launch_merge_t<64, true>(m, l, o, C, B, S_q, H, out, lse, s)
                             : launch_merge_t<64, false>(m, l, o, C, B, S_q, H, out, lse, s);
    case 128: return out_bf16 ? launch_merge_t<128, true>(m, l, o, C, B, S_q, H, out, lse, s)
                              : launch_merge_t<128, false>(m, l, o, C, B, S_q, H, out, lse, s);
    case 256: return out_bf16 ? launch_merge_t<256, true>(m, l, o, C, B, S_q, H, out, lse, s)
                              : launch_merge_t<256, false>(m, l, o, C, B, S_q, H, out, lse, s);
  }
  return ATTN_ERR_UNSUPPORTED;
}

unsigned int merge_take_status(cudaStream_t s) {
  if (cudaStreamSynchronize(s) != cudaSuccess) return kStatusTimeout;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_merge_status, sizeof(v)) != cudaSuccess) return kStatusTimeout;
  if (v != 0) {
    const unsigned int zero = 0;
    cudaMemcpyToSymbol(g_merge_status, &zero, sizeof(zero));
  }
  return v;
}

}  // namespace attn
