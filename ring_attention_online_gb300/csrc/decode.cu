// Split-KV decode partials: one query per sequence, a long KV read in place.
//
// "kernbench2 _attention_mesh_mlo.py": every rank keeps its sequence shard of
// KV in place and computes ONE local partial (m, l, o) of the replicated query
// against it; the triplets are then merged and normalised.  On one GPU the
// shards are num_splits chunks of ceil(S_kv / num_splits) keys; this kernel
// computes the partial of one (batch, KV head, chunk) for all G = h_q / h_kv
// query heads of the group, and merge.cu folds the chunks.  Where the page
// normalises o with a softmax before its merge, the partial here is the
// unnormalised sum exp(s - m) v that its merge and final o / l require.
//
// The kernel is HBM-bound (each K/V byte is read once): a producer warp streams
// 64-key K and V stages with TMA into a ring of shared-memory buffers; four
// consumer warps each take 16 keys of a stage.  Per warp, S = Q.K^T and
// O += P.V run on mma.sync m16n8k16 with the G query heads as the M rows
// (padded to 16); the S accumulator fragment is reused as the A fragment of
// P.V.  At the end the four warps' triplets are merged in shared memory.
//
// Fused merge (when `counters` is given): each CTA counts itself in its
// (batch, KV head) counter after its partials are written, and the last of the
// num_splits CTAs folds all chunks' partials of its G query heads into the
// final O and LSE, so no second kernel and no host round trip is needed.
#include <math_constants.h>

#include "common.cuh"
#include "checked.cuh"
#include "merge.cuh"
#include "ptx.cuh"

namespace attn {

static __device__ unsigned int g_decode_status;

template <int D>
struct DecodeCfg {
  static constexpr int KEYS = 64;                     // keys per stage
  static constexpr int BLOCK_BYTES = KEYS * 128;      // one TMA block: 64 keys x 64 columns
  static constexpr int TILE_BYTES = KEYS * D * 2;     // K (or V) of one stage
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int NST = D == 256 ? 2 : (96 * 1024) / STAGE_BYTES;
  static constexpr int SMEM_BYTES = NST * STAGE_BYTES + 1024;
  static constexpr int CONSUMERS = 4;
  static constexpr int THREADS = 32 * (CONSUMERS + 1);
  // end-of-CTA merge scratch (reuses the stage buffers): O [4][16][D] + m,l [4][16]
  static_assert(CONSUMERS * 16 * D * 4 + 2 * CONSUMERS * 16 * 4 <= NST * STAGE_BYTES, "merge scratch fits");
};

__device__ __forceinline__ bool dc_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort, uint32_t site) {
  if (mbar_try_wait(smem_u32(bar), parity)) return true;
  if (*reinterpret_cast<volatile unsigned int*>(&g_decode_status) & kStatusTimeout) {
    *abort = 1u;
    return false;
  }
  return mbar_wait_bounded(bar, parity, abort, &g_decode_status, kStatusTimeout | (site << kStatusSiteShift),
                           kWaitTimeoutNs);
}

__device__ __forceinline__ void dc_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (global_timer_ns() - t0 > kWaitTimeoutNs) {
      atomicOr(&g_decode_status, kStatusTimeout | (0x90u << kStatusSiteShift));
      return;
    }
  }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <bool kBf16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (kBf16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// Byte address of element (key, d) of a [64 keys x D] tile stored as D/64
// swizzled blocks of 64 keys x 128 bytes; d must be a multiple of 8.
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int key, int d) {
  return base + (d >> 6) * (64 * 128) + key * 128 + ((((d & 63) >> 3) ^ (key & 7)) << 4);
}

template <int D, bool kBf16>
__global__ void __launch_bounds__(160) decode_partial_kernel(const __grid_constant__ CUtensorMap mk,
                                                             const __grid_constant__ CUtensorMap mv,
                                                             const uint16_t* __restrict__ q, float* __restrict__ m_out,
                                                             float* __restrict__ l_out, float* __restrict__ o_out,
                                                             int B, int S_kv, int h_q, int h_kv, float c,
                                                             int num_splits, int* __restrict__ counters,
                                                             void* __restrict__ out, float* __restrict__ lse) {
  using C = DecodeCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[C::NST], bar_empty[C::NST];
  __shared__ uint32_t abort_flag;
  __shared__ int last_of_group;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int g = blockIdx.x;      // KV head (fastest: the heads of one token row are read together)
  const int split = blockIdx.y;
  const int b = blockIdx.z;
  const int G = h_q / h_kv;
  const int chunk = (S_kv + num_splits - 1) / num_splits;
  const long long lo_ll = (long long)split * chunk;
  const int k_lo = (int)(lo_ll < S_kv ? lo_ll : S_kv);
  const int k_hi = (int)(lo_ll + chunk < S_kv ? lo_ll + chunk : S_kv);
  const int ntiles = (k_hi - k_lo + C::KEYS - 1) / C::KEYS;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], C::CONSUMERS);
    }
    fence_barrier_init();
  }
  __syncthreads();

  // per consumer warp running triplet; rows 0..15 = query heads g*G + row
  const int gq = lane >> 2;  // fragment row (and row + 8)
  const int tq = lane & 3;
  float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};
  float l_run[2] = {0.f, 0.f};   // fp32 sum of exp2(x - m): the triplet's l
  float lr_run[2] = {0.f, 0.f};  // sum of the rounded P used by the MMA: normalises O
  float acc[D / 8][4];
  bool ok = true;

  if (warp == C::CONSUMERS) {
    // ============================================================ producer
    if (lane == 0 && ntiles > 0) {
      prefetch_tensormap(&mk);
      prefetch_tensormap(&mv);
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        if (!dc_wait(&bar_empty[stage], phase ^ 1u, &abort_flag, 1)) break;
        uint8_t* dst = smem + stage * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&bar_full[stage], C::STAGE_BYTES);
        const int key0 = k_lo + t * C::KEYS;
        for (int blk = 0; blk < D / 64; ++blk) {
          // a load whose coordinates fail the checked build's test loads tile 0
          const bool c_ok = check_tile(blk * 64, g, key0, b, D, h_kv, S_kv, B, C::KEYS, &g_decode_status);
          const int c0 = c_ok ? blk * 64 : 0, c1 = c_ok ? g : 0, c2 = c_ok ? key0 : 0, c3 = c_ok ? b : 0;
          tma_load_4d(dst + blk * C::BLOCK_BYTES, &mk, &bar_full[stage], c0, c1, c2, c3);
          tma_load_4d(dst + C::TILE_BYTES + blk * C::BLOCK_BYTES, &mv, &bar_full[stage], c0, c1, c2, c3);
        }
        ++issued;
        if (++stage == C::NST) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (abort_flag) {
        const int outstanding = issued < C::NST ? issued : C::NST;
        for (int i = 0; i < outstanding; ++i) {
          const int pos = issued - 1 - i;
          dc_drain(&bar_full[pos % C::NST], (uint32_t)((pos / C::NST) & 1));
        }
      }
    }
  } else {
    // ============================================================ consumers
    // Q as the A operand: rows = heads (zero beyond G), k = head dimension
    uint32_t qa[D / 16][4];
    {
      const int r0 = gq, r1 = gq + 8;
      const uint32_t* q0 = reinterpret_cast<const uint32_t*>(q + ((size_t)b * h_q + (size_t)g * G + r0) * D);
      const uint32_t* q1 = reinterpret_cast<const uint32_t*>(q + ((size_t)b * h_q + (size_t)g * G + r1) * D);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int c0 = (kk * 16 + 2 * tq) >> 1;
        const int c1 = (kk * 16 + 2 * tq + 8) >> 1;
        qa[kk][0] = r0 < G ? q0[c0] : 0u;
        qa[kk][1] = r1 < G ? q1[c0] : 0u;
        qa[kk][2] = r0 < G ? q0[c1] : 0u;
        qa[kk][3] = r1 < G ? q1[c1] : 0u;
      }
    }
#pragma unroll
    for (int i = 0; i < D / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    const int wkey = warp * 16;  // this warp's keys inside a stage
    const int mi = lane >> 3, mr = lane & 7;
    int stage = 0;
    uint32_t phase = 0;
    for (int t = 0; t < ntiles; ++t) {
      if (!dc_wait(&bar_full[stage], phase, &abort_flag, 2)) {
        ok = false;
        break;
      }
      const uint32_t kbase = smem_u32(smem + stage * C::STAGE_BYTES);
      const uint32_t vbase = kbase + C::TILE_BYTES;
      // S = Q . K^T for 16 keys: two n-tiles of 8 keys
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(tile_addr(kbase, wkey + (mi >> 1) * 8 + mr, kk * 16 + (mi & 1) * 8), b0, b1, b2, b3);
        mma16816<kBf16>(s0, qa[kk], b0, b1);
        mma16816<kBf16>(s1, qa[kk], b2, b3);
      }
      // keys of this warp: key0 + [2tq, 2tq+1] (s0) and key0 + 8 + [2tq, 2tq+1] (s1)
      const int key0 = k_lo + t * C::KEYS + wkey;
      const int lim = k_hi - key0;  // keys >= lim are outside this chunk
      if (lim < 16) {
        if (2 * tq >= lim) s0[0] = s0[2] = -CUDART_INF_F;
        if (2 * tq + 1 >= lim) s0[1] = s0[3] = -CUDART_INF_F;
        if (8 + 2 * tq >= lim) s1[0] = s1[2] = -CUDART_INF_F;
        if (8 + 2 * tq + 1 >= lim) s1[1] = s1[3] = -CUDART_INF_F;
      }
      // online softmax per row (row gq: elements 0,1; row gq+8: elements 2,3)
      float alpha[2];
      uint32_t pa[4];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float mx = fmaxf(fmaxf(s0[2 * r], s0[2 * r + 1]), fmaxf(s1[2 * r], s1[2 * r + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run[r], mx * c);
        const float ref = m_new == -CUDART_INF_F ? 0.f : m_new;
        alpha[r] = fast_exp2(m_run[r] - ref);  // 0 while m_run = -inf
        m_run[r] = m_new;
        const float p0 = fast_exp2(fmaf(s0[2 * r], c, -ref));
        const float p1 = fast_exp2(fmaf(s0[2 * r + 1], c, -ref));
        const float p2 = fast_exp2(fmaf(s1[2 * r], c, -ref));
        const float p3 = fast_exp2(fmaf(s1[2 * r + 1], c, -ref));
        pa[r] = pack_half2<kBf16>(p0, p1);      // a0,a1 / a2,a3: keys 2tq, 2tq+1
        pa[2 + r] = pack_half2<kBf16>(p2, p3);  // a4,a5 / a6,a7: keys 8+2tq, 8+2tq+1
        // lanes of a quad each hold a part of both sums
        const float2 ra = unpack_half2<kBf16>(pa[r]), rb = unpack_half2<kBf16>(pa[2 + r]);
        lr_run[r] = lr_run[r] * alpha[r] + ((ra.x + ra.y) + (rb.x + rb.y));
        l_run[r] = l_run[r] * alpha[r] + ((p0 + p1) + (p2 + p3));
      }
      // O = O * alpha + P . V
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(tile_addr(vbase, wkey + (mi & 1) * 8 + mr, np * 16 + (mi >> 1) * 8), b0, b1, b2, b3);
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          float* a = acc[2 * np + h2];
          a[0] *= alpha[0];
          a[1] *= alpha[0];
          a[2] *= alpha[1];
          a[3] *= alpha[1];
        }
        const uint32_t afrag[4] = {pa[0], pa[1], pa[2], pa[3]};
        mma16816<kBf16>(acc[2 * np], afrag, b0, b1);
        mma16816<kBf16>(acc[2 * np + 1], afrag, b2, b3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_empty[stage]);
      if (++stage == C::NST) {
        stage = 0;
        phase ^= 1u;
      }
    }
    // both sums are split across the 4 lanes of a quad
    float ratio[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
      lr_run[r] += __shfl_xor_sync(0xffffffffu, lr_run[r], 1);
      lr_run[r] += __shfl_xor_sync(0xffffffffu, lr_run[r], 2);
      ratio[r] = lr_run[r] > 0.f ? l_run[r] / lr_run[r] : 0.f;
    }
    // O re-weighted so that O / l equals the consistently normalised O_acc / lr
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      acc[nt][0] *= ratio[0];
      acc[nt][1] *= ratio[0];
      acc[nt][2] *= ratio[1];
      acc[nt][3] *= ratio[1];
    }
  }

  // ============================================================ CTA merge of the 4 warps
  __syncthreads();  // every stage consumed (or aborted); shared memory is free
  if (abort_flag) return;
  float* so = reinterpret_cast<float*>(smem);              // [4][16][D]
  float* sm = so + C::CONSUMERS * 16 * D;                  // [4][16]
  float* sl = sm + C::CONSUMERS * 16;                      // [4][16]
  if (warp < C::CONSUMERS) {
    float* ow = so + warp * 16 * D;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      const int d = nt * 8 + 2 * tq;
      *reinterpret_cast<float2*>(ow + gq * D + d) = make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2*>(ow + (gq + 8) * D + d) = make_float2(acc[nt][2], acc[nt][3]);
    }
    if (tq == 0) {
      sm[warp * 16 + gq] = m_run[0];
      sm[warp * 16 + gq + 8] = m_run[1];
      sl[warp * 16 + gq] = l_run[0];
      sl[warp * 16 + gq + 8] = l_run[1];
    }
  }
  __syncthreads();
  // rows 0..G-1 x D columns over all 160 threads
  constexpr float kLn2 = 0.693147180559945309f;
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int r = idx / D, d = idx % D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < C::CONSUMERS; ++w) M = fmaxf(M, sm[w * 16 + r]);
    float o = 0.f, l = 0.f;
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < C::CONSUMERS; ++w) {
        const float mw = sm[w * 16 + r];
        const float f = mw == -CUDART_INF_F ? 0.f : fast_exp2(mw - M);
        o += f * so[(w * 16 + r) * D + d];
        l += f * sl[w * 16 + r];
      }
    }
    const size_t row = ((size_t)split * B + b) * h_q + (size_t)g * G + r;  // [C, B, h_q]
    if (!check_index((long long)row, (long long)num_splits * B * h_q, &g_decode_status)) continue;
    o_out[row * D + d] = o;
    if (d == 0) {
      m_out[row] = M == -CUDART_INF_F ? -CUDART_INF_F : M * kLn2;
      l_out[row] = l;
    }
  }
  (void)ok;
  if (counters == nullptr) return;

  // ============================================================ fused merge
  __threadfence();  // this CTA's partials are visible device-wide before it is counted
  __syncthreads();
  if (!check_index((long long)b * h_kv + g, (long long)B * h_kv, &g_decode_status)) return;
  int* counter = counters + (size_t)b * h_kv + g;
  if (threadIdx.x == 0) last_of_group = atomicAdd(counter, 1) == num_splits - 1;
  __syncthreads();
  if (!last_of_group) return;
  __threadfence();  // the partials of the CTAs counted before this one are visible
  const size_t ml_stride = (size_t)B * h_q;
  for (int r = warp; r < G; r += C::CONSUMERS + 1) {
    const size_t hrow = (size_t)b * h_q + (size_t)g * G + r;  // [B, h_q]: O is [B, h_q, D]
    merge_row<D, kBf16>(m_out, l_out, o_out, num_splits, ml_stride, hrow, ml_stride * D, hrow * D, out, lse, hrow,
                        lane, (long long)B * h_q, &g_decode_status);
  }
  if (threadIdx.x == 0) *counter = 0;  // ready for the next call on this workspace
}

template <int D, bool kBf16>
static attn_status_t launch_decode_t(const void* q, const CUtensorMap& mk, const CUtensorMap& mv, float* m, float* l,
                                     float* o, int B, int S_kv, int h_q, int h_kv, float c, int num_splits,
                                     int* counters, void* out, float* lse, cudaStream_t s) {
  using C = DecodeCfg<D>;
  auto kern = decode_partial_kernel<D, kBf16>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const dim3 grid(h_kv, num_splits, B);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, s>>>(mk, mv, static_cast<const uint16_t*>(q), m, l, o, B, S_kv, h_q, h_kv,
                                                c, num_splits, counters, out, lse);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t launch_decode_partial(const void* q, const CUtensorMap& mk, const CUtensorMap& mv, float* m, float* l,
                                    float* o, int B, int S_kv, int h_q, int h_kv, int D, bool bf16, float scale_log2,
                                    int num_splits, int* counters, void* out, float* lse, cudaStream_t s) {
#define ATTN_DECODE_CASE(DD)                                                                                     \
  case DD:                                                                                                       \
    return bf16 ? launch_decode_t<DD, true>(q, mk, mv, m, l, o, B, S_kv, h_q, h_kv, scale_log2, num_splits,     \
                                            counters, out, lse, s)                                               \
                : launch_decode_t<DD, false>(q, mk, mv, m, l, o, B, S_kv, h_q, h_kv, scale_log2, num_splits,    \
                                             counters, out, lse, s);
  switch (D) {
    ATTN_DECODE_CASE(64)
    ATTN_DECODE_CASE(128)
    ATTN_DECODE_CASE(256)
  }
#undef ATTN_DECODE_CASE
  return ATTN_ERR_UNSUPPORTED;
}

unsigned int decode_take_status(cudaStream_t s) {
  if (cudaStreamSynchronize(s) != cudaSuccess) return kStatusTimeout;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_decode_status, sizeof(v)) != cudaSuccess) return kStatusTimeout;
  if (v != 0) {
    const unsigned int zero = 0;
    cudaMemcpyToSymbol(g_decode_status, &zero, sizeof(zero));
  }
  return v;
}

}  // namespace attn
