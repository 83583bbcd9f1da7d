// Fold of C partial triplets per row, then the final normalisation.
//
// "kernbench2 _gqa_prefill_long.py" (online-softmax merge into the running
// (m, l, O); final normalise O / l) and "kernbench2 _attention_mesh_mlo.py"
// (merge-from-W / merge-from-E of (m, l, o) triplets; final normalize).
// Folding C triplets pairwise with m_new = max(m, m_s) equals, up to rounding,
// one pass with the global max M = max_c m_c:
//   l = sum_c l_c exp(m_c - M),  O = sum_c o_c exp(m_c - M) / l,  LSE = M + ln l.
// Empty partials (m_c = -inf) get weight 0, never NaN.
//
// One warp per output row; each lane owns D/32 contiguous columns, so every
// partial row is read once with coalesced 8..32-byte loads.  HBM-bound.
#include <math_constants.h>

#include "common.cuh"
#include "ptx.cuh"

namespace attn {

template <int D, bool kBf16>
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ m, const float* __restrict__ l,
                                                    const float* __restrict__ o, int C, int B, int S_q, int H,
                                                    void* __restrict__ out, float* __restrict__ lse) {
  constexpr int PER = D / 32;
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
  const size_t ml_stride = (size_t)B * H * S_q;
  const size_t ml_idx = ((size_t)b * H + h) * S_q + s;
  const size_t o_stride = (size_t)rows * D;
  const size_t o_idx = (size_t)row * D + (size_t)lane * PER;

  float M = -CUDART_INF_F;
  for (int c = lane; c < C; c += 32) M = fmaxf(M, m[c * ml_stride + ml_idx]);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, d));

  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  float lsum = 0.f;
  if (M != -CUDART_INF_F) {
    constexpr float kLog2e = 1.4426950408889634f;
    for (int c0 = 0; c0 < C; c0 += 32) {
      const int c = c0 + lane;
      float w = 0.f;
      if (c < C) {
        const float mc = m[c * ml_stride + ml_idx];
        w = mc == -CUDART_INF_F ? 0.f : exp2f((mc - M) * kLog2e);
        lsum += w * l[c * ml_stride + ml_idx];
      }
      const int cnt = min(32, C - c0);
      for (int cc = 0; cc < cnt; ++cc) {
        const float wc = __shfl_sync(0xffffffffu, w, cc);
        if (wc == 0.f) continue;  // uniform across the warp
        const float* src = o + (size_t)(c0 + cc) * o_stride + o_idx;
        if constexpr (PER == 2) {
          const float2 x = *reinterpret_cast<const float2*>(src);
          acc[0] = fmaf(wc, x.x, acc[0]);
          acc[1] = fmaf(wc, x.y, acc[1]);
        } else {
#pragma unroll
          for (int v4 = 0; v4 < PER / 4; ++v4) {
            const float4 x = reinterpret_cast<const float4*>(src)[v4];
            acc[4 * v4 + 0] = fmaf(wc, x.x, acc[4 * v4 + 0]);
            acc[4 * v4 + 1] = fmaf(wc, x.y, acc[4 * v4 + 1]);
            acc[4 * v4 + 2] = fmaf(wc, x.z, acc[4 * v4 + 2]);
            acc[4 * v4 + 3] = fmaf(wc, x.w, acc[4 * v4 + 3]);
          }
        }
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, d);
  }
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  uint32_t packed[PER / 2];
#pragma unroll
  for (int i = 0; i < PER / 2; ++i) packed[i] = pack_half2<kBf16>(acc[2 * i] * inv, acc[2 * i + 1] * inv);
  uint16_t* dst = reinterpret_cast<uint16_t*>(out) + o_idx;
  if constexpr (PER == 2) {
    *reinterpret_cast<uint32_t*>(dst) = packed[0];
  } else if constexpr (PER == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  } else {
    *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
  if (lse != nullptr && lane == 0) lse[ml_idx] = lsum > 0.f ? M + logf(lsum) : -CUDART_INF_F;
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

}  // namespace attn
