// Fold of C partial triplets of one row, then the final normalisation; shared
// by the merge kernel and the decode kernel's fused tail.
//
// "kernbench2 _gqa_prefill_long.py" (online-softmax merge into the running
// (m, l, O); final normalise O / l) and "kernbench2 _attention_mesh_mlo.py"
// (merge-from-W / merge-from-E of (m, l, o) triplets; final normalize).
// Folding C triplets pairwise with m_new = max(m, m_s) equals, up to rounding,
// one pass with the global max M = max_c m_c:
//   l = sum_c l_c exp(m_c - M),  O = sum_c o_c exp(m_c - M) / l,  LSE = M + ln l.
// Empty partials (m_c = -inf) get weight 0, never NaN.
#pragma once

#include <math_constants.h>

#include "checked.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace attn {

// One warp folds one row.  Partial c of the row: m[c * ml_stride + ml_idx],
// l[...] (natural-log units), o[c * o_stride + o_idx .. + D).  Each lane owns
// D/32 contiguous columns, so every partial row is read once with coalesced
// loads; the loads bypass L1 because the partials may have been written by
// other CTAs of the same kernel.
// out_rows: rows of `out` (and of `lse`); status: the calling kernel's status
// word, for the checked build's store checks.
template <int D, bool kBf16>
__device__ __forceinline__ void merge_row(const float* __restrict__ m, const float* __restrict__ l,
                                          const float* __restrict__ o, int C, size_t ml_stride, size_t ml_idx,
                                          size_t o_stride, size_t o_idx, void* __restrict__ out,
                                          float* __restrict__ lse, size_t lse_idx, int lane, long long out_rows,
                                          unsigned int* status) {
  constexpr int PER = D / 32;
  const size_t col = o_idx + (size_t)lane * PER;
  float M = -CUDART_INF_F;
  for (int c = lane; c < C; c += 32) M = fmaxf(M, __ldcg(m + c * ml_stride + ml_idx));
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
        const float mc = __ldcg(m + c * ml_stride + ml_idx);
        w = mc == -CUDART_INF_F ? 0.f : exp2f((mc - M) * kLog2e);
        lsum += w * __ldcg(l + c * ml_stride + ml_idx);
      }
      const int cnt = min(32, C - c0);
      // four partial rows in flight per step; a zero weight (an empty
      // partial) leaves the sum untouched whatever its O holds
      for (int cc = 0; cc < cnt; cc += 4) {
        float wv[4];
        float x[4][PER];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          wv[u] = __shfl_sync(0xffffffffu, w, (cc + u) & 31);
          if (cc + u >= cnt) wv[u] = 0.f;
          const float* src = o + (size_t)(c0 + (cc + u < cnt ? cc + u : cc)) * o_stride + col;
          if constexpr (PER == 2) {
            const float2 v2 = __ldcg(reinterpret_cast<const float2*>(src));
            x[u][0] = v2.x;
            x[u][1] = v2.y;
          } else {
#pragma unroll
            for (int v4 = 0; v4 < PER / 4; ++v4) {
              const float4 v = __ldcg(reinterpret_cast<const float4*>(src) + v4);
              x[u][4 * v4 + 0] = v.x;
              x[u][4 * v4 + 1] = v.y;
              x[u][4 * v4 + 2] = v.z;
              x[u][4 * v4 + 3] = v.w;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int i = 0; i < PER; ++i) acc[i] = wv[u] != 0.f ? fmaf(wv[u], x[u][i], acc[i]) : acc[i];
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, d);
  }
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  uint32_t packed[PER / 2];
#pragma unroll
  for (int i = 0; i < PER / 2; ++i) packed[i] = pack_half2<kBf16>(acc[2 * i] * inv, acc[2 * i + 1] * inv);
  uint16_t* dst = reinterpret_cast<uint16_t*>(out) + col;
  if (!check_index((long long)(col / D), out_rows, status) || !check_index((long long)lse_idx, out_rows, status))
    return;
  if constexpr (PER == 2) {
    *reinterpret_cast<uint32_t*>(dst) = packed[0];
  } else if constexpr (PER == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  } else {
    *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
  if (lse != nullptr && lane == 0) lse[lse_idx] = lsum > 0.f ? M + logf(lsum) : -CUDART_INF_F;
}

}  // namespace attn
