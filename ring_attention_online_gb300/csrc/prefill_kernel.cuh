// Blockwise online-softmax attention forward, tcgen05 + TMA, Q tiles of 128
// rows, persistent over units of two for dense launches.
//
// What it computes, by source:
//  * "kernbench2 _gqa_prefill_long.py", gqa_prefill_long_kernel: per KV block,
//    scores = Q.K^T, m = rowmax, exp(scores - m), l = rowsum, O = exp . V; each
//    block merged into the running (m, l, O) with m_new = max(m, m_step) and the
//    factors exp(m - m_new), exp(m_step - m_new); at the end O / l.  Here the
//    "blocks" are 128-key tiles and the running triplet lives in registers (m, l)
//    and TMEM (O); the page's ring steps become a ring-order walk over chunks.
//  * "[pallas] Support dependent Tile.end bounds in Pallas": the tile walk ends
//    at min(kv_end, tile_q.end) (no fully masked tile is visited); only the
//    diagonal and tail tiles are masked.
//
// Work: dense, partial and window launches run one CTA per SM over units of
// two Q tiles of one (batch, head), t and n_qt - 1 - t when causal (so every
// unit walks n_qt + 1 KV tiles) or 2x and 2x + 1 otherwise, the longer first;
// a jagged CTA takes one worklist item.  Barrier phases and the K/V stage rings
// run on across all of a CTA's items, so each item's Q and first K/V tiles
// load, and its first S is computed, while the previous item's last tiles and
// epilogue finish: with one CTA per Q tile, a CTA's fixed costs (start-up,
// first loads, pipeline fill and drain) were ~11 K cycles, 18 % of the dense
// causal S=4096 launch.
//
// CTA layout (352 threads):
//   warp 0      TMA producer: per item the Q tile (once the previous item's S
//               MMAs are done with the Q buffer), then K/V 128-column slabs
//               through a K ring and a V ring of shared-memory stages, in
//               the order K(0), then per tile K(j+1), V(j).
//   warp 1      TMEM owner and S issuer: S(j) = Q.K_j^T into the one
//               128-column S buffer, once the softmax warps have read S(j-1)
//               out of it.
//   warp 10     PV issuer: O += P(j).V_j, P(j) (bf16/fp16, written by the
//               softmax warps to P buffer j mod 2) being the TMEM A operand.
//   warps 2..9  softmax + epilogue: each query row (TMEM lane) is shared by two
//               warps, one per half of the tile's 128 keys and of O's columns.
//               Scores are scaled into the exp2 domain; the running max is
//               raised lazily (only when it grows by more than 2^8), so O is
//               rescaled in TMEM only on those tiles - the result is the same
//               up to rounding because l and O always share one reference max.
//
// Every wait is bounded (see pf_wait); a timeout sets the library's device
// status, the CTA skips its remaining work, drains its copies and MMAs and
// frees TMEM before returning.
#pragma once

#include <math_constants.h>

#include "prefill_common.cuh"

namespace attn {

template <int D>
struct PrefillCfg {
  static constexpr int BM = 128;
  static constexpr int BN = 128;
  static constexpr int SC = D < 128 ? D : 128;  // columns per K/V slab (one smem stage)
  static constexpr int NH = D / SC;             // slabs per K or V tile
  static constexpr int BLK_PER_SLAB = SC / 64;  // 64-column TMA blocks per slab
  static constexpr int BLOCK_BYTES = 128 * 128; // one TMA block: 128 rows x 128 bytes
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int SLAB_BYTES = BN * SC * 2;
  // four K/V slabs in flight: on GB300 two to six stages time the same, so
  // the rest of shared memory stays free for the softmax warps' exchanges.
  // K and V have rings of their own (NST / 2 stages each, K first), so each
  // stage's fills are consumed by one issuer in order: a consumer never waits
  // on a fill while the stage's previous one is still pending, which the
  // parity wait of an mbarrier could not tell from a completed one
  static constexpr int NST = D == 64 ? 8 : 4;
  static constexpr int RING = NST / 2;  // stages per ring
  static constexpr int SMEM_BYTES = Q_BYTES + NST * SLAB_BYTES + 1024;  // + 1 KB alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  // TMEM: S(j) in columns [0, 128) (one buffer); P(j) (bf16/fp16, 64 columns)
  // in [P_COL + 64*(j%2), +64); O in [O_COL, O_COL + D)
  static constexpr uint32_t P_COL = 128;
  static constexpr uint32_t O_COL = 256;
  static constexpr int THREADS = 352;  // TMA warp, S issuer, 8 softmax warps, PV issuer
  static_assert(D == 64 || D == 128 || D == 256, "head dim");
  static_assert(NST >= 2 && NST % 2 == 0, "K and V rings of equal size");
  static_assert(O_COL + D <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// kOneChunk: the launch walks a single chunk (no ring order); the literal lets
// the compiler drop the ring-order walk state
template <int D, bool kBf16, int kMode, bool kOneChunk>
__global__ void __launch_bounds__(352, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mv, const PrefillParams p) {
  using C = PrefillCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_q, bar_qe, bar_fin;  // Q landed; Q buffer free (the item's S MMAs done)
  __shared__ uint64_t bar_o[2];  // PV(j) completes a phase of bar_o[j % 2]
  __shared__ uint64_t bar_full[C::NST], bar_empty[C::NST];
  __shared__ uint64_t bar_s[2], bar_p[2];
  __shared__ uint64_t bar_sfree[2];  // the softmax warps have read S(j) out of TMEM (j % 2)
  __shared__ uint32_t tmem_slot;
  __shared__ uint32_t abort_flag;
  __shared__ float xch_max[2][2][128];  // [tile parity][column half][row]
  __shared__ float xch_l[2][2][128], xch_lr[2][2][128];  // [item parity][column half][row]
  __shared__ uint64_t bar_x[2][4];       // pair exchange barriers: [tile parity][lane quarter]
  __shared__ uint64_t bar_xe[4];         // end-of-row exchange barrier per lane quarter

  // ------------------------------------------------------------ work items
  // Dense / window / partial launches are persistent: CTA c takes the units
  // c, c + grid, c + 2 grid, ... in the order (pair x, head, batch), so the
  // CTAs running at one time share the K/V of a few heads in L2.  A unit is
  // two Q tiles of one (batch, head), t and n_qt - 1 - t when causal (every
  // unit then walks n_qt + 1 KV tiles; the longer first), 2x and 2x + 1
  // otherwise; its second slot is empty when the two coincide or the second
  // lies past the end.  Barrier phases and the stage rings run on across all of
  // a CTA's items, so each item's Q and first K/V tiles load, and its first S
  // is computed, while the previous item finishes.  One CTA per unit (the
  // hardware's launch order) measured 4 % slower: the CTA start-up and
  // pipeline fill and drain were exposed once per unit.  Jagged launches take
  // one worklist item per CTA.
  struct Item {
    int b, h, q_lo, q_hi, kv_lo, kv_hi, q_pos0, kv_pos0;
    bool valid;
  };
  const int n_qt = (p.S_q + C::BM - 1) / C::BM;
  const int n_ux = (n_qt + 1) / 2;  // units per (batch, head)
  int n_my = 1;                     // item slots of this CTA
  if constexpr (kMode == kModeJagged) {
    if ((int)blockIdx.x >= *p.work_count) return;  // the grid is an upper bound on the item count
  } else {
    const long long units = (long long)n_ux * p.h_q * p.B;
    n_my = 2 * (int)((units - (long long)blockIdx.x + gridDim.x - 1) / gridDim.x);
  }
  auto get_item = [&](int i) -> Item {
    Item it;
    it.valid = true;
    if constexpr (kMode == kModeJagged) {
      (void)i;
      const int4 w = p.work_items[blockIdx.x];
      it.b = 0;
      it.h = blockIdx.y;
      it.q_lo = w.z;
      it.q_hi = w.z + w.w;
      it.kv_lo = w.x;
      it.kv_hi = w.x + w.y;  // seq_offsets[seq_idx + 1]
      it.q_pos0 = 0;
      it.kv_pos0 = 0;
    } else {
      const long long u = (long long)blockIdx.x + (long long)(i >> 1) * gridDim.x;
      const int x = (int)(u % n_ux);
      const long long yb = u / n_ux;
      int qt;
      if (p.causal) {
        const int t_first = n_qt - 1 - x;
        qt = (i & 1) ? x : t_first;
        it.valid = !(i & 1) || x < t_first;
      } else {
        qt = 2 * x + (i & 1);
        it.valid = qt < n_qt;
      }
      it.b = (int)(yb / p.h_q);
      it.h = (int)(yb % p.h_q);
      it.q_lo = qt * C::BM;
      it.q_hi = min(it.q_lo + C::BM, p.S_q);
      it.kv_lo = p.kv_lo;
      it.kv_hi = p.kv_hi;
      it.q_pos0 = p.q_pos0;
      it.kv_pos0 = p.kv_pos0;
    }
    return it;
  };
  auto item_walk = [&](const Item& it, TileWalk& w) -> int {
    w.init(it.q_lo, it.q_hi, it.kv_lo, it.kv_hi, it.q_pos0, it.kv_pos0, p.causal, kOneChunk ? 1 : p.num_chunks, C::BN,
           kMode == kModeWindow ? p.window : -1);
    return w.count();
  };
  int hk = (int)blockIdx.y / p.group;  // the producer's KV head, set per item

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + C::Q_BYTES;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_q, 1);
    mbar_init(&bar_qe, 1);
    mbar_init(&bar_o[0], 1);
    mbar_init(&bar_o[1], 1);
    mbar_init(&bar_fin, 2);  // one commit per MMA issuer
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_s[i], 1);
      mbar_init(&bar_sfree[i], 256);
      mbar_init(&bar_p[i], 256);
      for (int q4 = 0; q4 < 4; ++q4) mbar_init(&bar_x[i][q4], 64);
    }
    for (int q4 = 0; q4 < 4; ++q4) mbar_init(&bar_xe[q4], 64);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    // ========================================================== TMA producer
    if (lane == 0) {
      prefetch_tensormap(&mq);
      prefetch_tensormap(&mk);
      prefetch_tensormap(&mv);
      int filled[2] = {0, 0};  // slabs issued into the K ring and the V ring
      int q_loads = 0;
      bool ok = true;
      // fill f of a ring goes to its stage f % RING; fill f - RING of that
      // stage must have been released by its issuer first
      auto push = [&](const CUtensorMap* map, int start, int bb, int ring) -> bool {
        int& fills = filled[ring];
        for (int hs = 0; hs < C::NH; ++hs, ++fills) {
          const int stage = ring * C::RING + fills % C::RING;
          const uint32_t phase = (uint32_t)((fills / C::RING) & 1);
          if (!pf_wait_outlined(&bar_empty[stage], phase ^ 1u, &abort_flag, 1)) return false;
          uint8_t* dst = sKV + stage * C::SLAB_BYTES;
          mbar_arrive_expect_tx(&bar_full[stage], C::SLAB_BYTES);
          for (int blk = 0; blk < C::BLK_PER_SLAB; ++blk)
            tma_load_4d(dst + blk * C::BLOCK_BYTES, map, &bar_full[stage], hs * C::SC + blk * 64, hk, start, bb);
        }
        return true;
      };
      for (int i = 0; ok && i < n_my; ++i) {
        const Item it = get_item(i);
        if (!it.valid) continue;
        hk = it.h / p.group;
        TileWalk walk;
        const int n = item_walk(it, walk);
        if (n == 0) continue;
        // the Q buffer is free once the previous item's S MMAs are done
        if (q_loads > 0 && !pf_wait_outlined(&bar_qe, (uint32_t)((q_loads - 1) & 1), &abort_flag, 13)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bar_q, C::Q_BYTES);
        for (int blk = 0; blk < D / 64; ++blk)
          tma_load_4d(sQ + blk * C::BLOCK_BYTES, &mq, &bar_q, blk * 64, it.h, it.q_lo, it.b);
        ++q_loads;
        TileWalk kw = walk, vw = walk;
        int ch, st, me;
        kw.next(ch, st, me);
        ok = push(&mk, st, it.b, 0);
        for (int j = 0; ok && j < n; ++j) {
          if (j + 1 < n) {
            kw.next(ch, st, me);
            ok = push(&mk, st, it.b, 0);
            if (!ok) break;
          }
          vw.next(ch, st, me);
          ok = push(&mv, st, it.b, 1);
        }
      }
      if (abort_flag) {
        // copies may still be landing in shared memory: wait for them
        if (q_loads > 0) pf_drain(&bar_q, (uint32_t)((q_loads - 1) & 1));
        for (int ring = 0; ring < 2; ++ring) {
          const int outstanding = filled[ring] < C::RING ? filled[ring] : C::RING;
          for (int i = 0; i < outstanding; ++i) {
            const int pos = filled[ring] - 1 - i;
            pf_drain(&bar_full[ring * C::RING + pos % C::RING], (uint32_t)((pos / C::RING) & 1));
          }
        }
      }
    }
  } else if (warp == 1 || warp == 10) {
    // ========================================================== MMA issuers
    // Warp 1 issues S(j), warp 10 issues PV(j).  A thread's wait stalls until
    // the tcgen05 work it issued itself has drained from the tensor pipe, so
    // with one issuer every wait (for P, or for a K/V stage) emptied the pipe.
    // Split by kind, each issuer only waits on work of the other roles: the S
    // issuer on K stages and on PV(j-2) (S(j) overwrites P(j-2) in its TMEM
    // buffer, and MMAs of different threads are not ordered), the PV issuer on
    // P(j) and V stages.
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_f16_f32acc(128, 128, kBf16, false);
      constexpr uint32_t kIdescPV = idesc_f16_f32acc(128, C::SC, kBf16, true);
      const uint32_t skv = smem_u32(sKV);
      // the S issuer takes every K slab, the PV issuer every V slab, each in
      // the order the producer filled its ring: slab f of a ring is in stage
      // ring * RING + f % RING, fill parity (f / RING) & 1.  Each slab is waited
      // for right before its MMAs, so the first half of S(j) (PV(j)) can run
      // while the second half's K (V) is still landing
      auto wait_slab = [&](int ring, int f, uint32_t site) -> bool {
        if (!pf_wait_outlined(&bar_full[ring * C::RING + f % C::RING], (uint32_t)((f / C::RING) & 1), &abort_flag,
                              site))
          return false;
        tc_fence_after_sync();
        return true;
      };
      bool ok = true;
      int g = 0;          // S (or PV) groups issued so far, all items: its barrier phases
      int slab_base = 0;  // slabs of this issuer's ring taken by the earlier items
      int q_used = 0;     // Q tiles consumed (S issuer)
      for (int i = 0; ok && i < n_my; ++i) {
        const Item it = get_item(i);
        if (!it.valid) continue;
        TileWalk walk;
        const int n = item_walk(it, walk);
        if (n == 0) continue;
        if (warp == 1) {
          const uint64_t qdesc = smem_desc_sw128(smem_u32(sQ), 16, 1024);
          ok = pf_wait_outlined(&bar_q, (uint32_t)(q_used & 1), &abort_flag, 5);
          tc_fence_after_sync();
          ++q_used;
          for (int j = 0; ok && j < n; ++j, ++g) {
            if (g >= 1) {
              // the one S buffer is free once the softmax warps have read the previous S
              ok = pf_wait_outlined(&bar_sfree[(g - 1) & 1], (uint32_t)(((g - 1) >> 1) & 1), &abort_flag, 11);
              if (!ok) break;
              tc_fence_after_sync();
            }
            const uint32_t d_tmem = tmem;
            for (int hs = 0; hs < C::NH; ++hs) {
              const int sl = slab_base + j * C::NH + hs;
              const int stage = sl % C::RING;  // K ring
              ok = wait_slab(0, sl, 2);
              if (!ok) break;
              const uint64_t kdesc = smem_desc_sw128(skv + stage * C::SLAB_BYTES, 16, 1024);
#pragma unroll
              for (int ks = 0; ks < C::SC / 16; ++ks) {
                const uint32_t qoff = (hs * C::BLK_PER_SLAB + ks / 4) * C::BLOCK_BYTES + (ks % 4) * 32;
                const uint32_t koff = (ks / 4) * C::BLOCK_BYTES + (ks % 4) * 32;
                mma_ss(d_tmem, desc_advance(qdesc, qoff), desc_advance(kdesc, koff), kIdescS, (hs | ks) != 0);
              }
              mma_commit(&bar_empty[stage]);
            }
            if (!ok) break;
            mma_commit(&bar_s[g & 1]);
          }
          // the item's S MMAs, the last readers of its Q, release the Q buffer
          if (ok) mma_commit(&bar_qe);
        } else {
          for (int j = 0; ok && j < n; ++j, ++g) {
            ok = pf_wait_outlined(&bar_p[g & 1], (uint32_t)((g >> 1) & 1), &abort_flag, 3);
            if (!ok) break;
            tc_fence_after_sync();  // P in TMEM
            const uint32_t p_tmem = tmem + C::P_COL + static_cast<uint32_t>((g & 1) * 64);
            const uint32_t acc0 = j > 0 ? 1u : 0u;  // the item's first PV starts O afresh
            for (int hs = 0; hs < C::NH; ++hs) {
              const int sl = slab_base + j * C::NH + hs;
              const int stage = C::RING + sl % C::RING;  // V ring
              ok = wait_slab(1, sl, 4);
              if (!ok) break;
              const uint64_t vdesc = smem_desc_sw128(skv + stage * C::SLAB_BYTES, 16384, 1024);
#pragma unroll
              for (int ks = 0; ks < C::BN / 16; ++ks)
                mma_ts(tmem + C::O_COL + hs * C::SC, p_tmem + ks * 8, desc_advance(vdesc, ks * 2048), kIdescPV,
                       ks > 0 ? 1u : acc0);
              mma_commit(&bar_empty[stage]);
            }
            if (!ok) break;
            mma_commit(&bar_o[g & 1]);
          }
        }
        slab_base += n * C::NH;
      }
      // every MMA either issuer issued must finish before TMEM is released
      mma_commit(&bar_fin);
      pf_drain(&bar_fin, 0);
    }
  } else {
    // ========================================================== softmax + epilogue
    // Two warps share each TMEM lane quarter: warp (2 + wq) and (6 + wq) ... take
    // the two column halves of every row (keys [64*half, 64*half + 64) of a tile,
    // O columns [half*D/2, half*D/2 + D/2)).  The pair exchanges row maxima once per
    // tile through shared memory, so both halves take identical decisions.
    const int sw = warp - 2;  // 0..7
    const int wq = warp & 3;  // TMEM lane quarter this warp may access
    const int half = sw >> 2;
    const int row = wq * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    constexpr int HD = D / 2;                                    // O columns per half
    const float c = p.scale_log2;  // > 0
    bool ok = true;
    int gj = 0;    // tiles so far, all items: the phases of the per-tile barriers
    int n_ep = 0;  // epilogues so far
    for (int i = 0; ok && i < n_my; ++i) {
      const Item it = get_item(i);
      if (!it.valid) continue;
      TileWalk sw_walk;
      const int n = item_walk(it, sw_walk);
      const int b = it.b, h = it.h, q_lo = it.q_lo, q_hi = it.q_hi, q_pos0 = it.q_pos0, kv_pos0 = it.kv_pos0;
      const int q_row = q_lo + row;
      float m_run = -CUDART_INF_F;   // reference max (exp2 domain), raised lazily
      float l_run = 0.f;             // this half's sum of exp2(x - m_run) in fp32: l and LSE
      float lr_run = 0.f;            // this half's sum of the rounded P the MMA multiplies V by
      float m_max = -CUDART_INF_F;   // true running max (partial mode)
      for (int j = 0; j < n; ++j, ++gj) {
        int ch, kstart, mend;
        sw_walk.next(ch, kstart, mend);
        const int buf = gj & 1;
        if (!pf_wait_outlined(&bar_s[buf], (uint32_t)((gj >> 1) & 1), &abort_flag, 6)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint32_t r0[32], r1[32];
        tmem_ld32(lane_addr + half * 64, r0);
        tmem_ld32(lane_addr + half * 64 + 32, r1);
        tmem_ld_wait(r0);
        tmem_ld_wait(r1);
        // S(j) is in registers: the S issuer may overwrite the buffer with S(j+1)
        tc_fence_before_sync();
        mbar_arrive(&bar_sfree[buf]);

        // mask the diagonal / tail tile (key kstart + i is visible iff i < lim)
        // and, under a sliding window, the tiles at its lower edge (iff i >= flo)
        constexpr bool win = kMode == kModeWindow;
        const bool need_mask =
            (kstart + C::BN > mend) ||
            (p.causal && ((long long)kv_pos0 + kstart + C::BN - 1 > (long long)q_pos0 + q_lo)) ||
            (win && (long long)kv_pos0 + kstart < (long long)q_pos0 + q_hi - 1 - p.window);
        if (need_mask) {
          long long lim = (long long)mend - kstart;
          long long flo = 0;
          if (p.causal) {
            const long long lc = (long long)q_pos0 + q_row - kv_pos0 - kstart + 1;
            lim = lc < lim ? lc : lim;
            if (win) flo = lc - 1 - p.window;
          }
          const long long lh = lim - half * 64, fh = flo - half * 64;  // limits within this half
          const uint32_t ninf = __float_as_uint(-CUDART_INF_F);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (i >= lh || i < fh) r0[i] = ninf;
            if (i + 32 >= lh || i + 32 < fh) r1[i] = ninf;
          }
        }
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          mx8[i] = fmax3(__uint_as_float(r0[i]), __uint_as_float(r0[i + 8]), __uint_as_float(r0[i + 16]));
          mx8[i] = fmax3(mx8[i], __uint_as_float(r0[i + 24]), __uint_as_float(r1[i]));
          mx8[i] = fmax3(mx8[i], __uint_as_float(r1[i + 8]), __uint_as_float(r1[i + 16]));
          mx8[i] = fmaxf(mx8[i], __uint_as_float(r1[i + 24]));
        }
        float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
        // both halves of the row see each other's max
        xch_max[buf][half][row] = mx;
        mbar_arrive(&bar_x[buf][wq]);
        if (!pf_wait_outlined(&bar_x[buf][wq], (uint32_t)((gj >> 1) & 1), &abort_flag, 9)) {
          ok = false;
          break;
        }
        mx = fmaxf(mx, xch_max[buf][half ^ 1][row]);
        const float m_tile = mx * c;  // -inf when the whole row is masked
        if constexpr (kMode == kModePartial) m_max = fmaxf(m_max, m_tile);
        const float m_new = fmaxf(m_run, m_tile);
        const bool raise = (m_new - m_run) > 8.0f;  // false when both are -inf
        float alpha = 1.f;
        if (raise) {
          alpha = fast_exp2(m_run - m_new);  // 0 on the first visible tile
          m_run = m_new;
          l_run *= alpha;
          lr_run *= alpha;
        }
        // P goes to P buffer gj % 2, which the PV two tiles back read; that PV is
        // waited for here and so always before this tile's PV is issued (no
        // waiter falls two phases behind on bar_o)
        if (gj >= 2) {
          if (!pf_wait_outlined(&bar_o[buf], (uint32_t)(((gj - 2) >> 1) & 1), &abort_flag, 12)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
        }
        const uint32_t pcol = lane_addr + C::P_COL + static_cast<uint32_t>(buf * 64);
        const float neg_m = m_run == -CUDART_INF_F ? 0.f : -m_run;
        const uint64_t c2 = f2_make(c, c), nm2 = f2_make(neg_m, neg_m);
        uint64_t sum2 = f2_make(0.f, 0.f);
        float sr[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // rounded weights, 8 chains
        uint32_t pk[16];
        auto pack_chunk = [&](uint32_t (&r)[32], uint32_t col) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 e = f2_split(f2_fma(f2_make_u(r[2 * i], r[2 * i + 1]), c2, nm2));
            const float p0 = fast_exp2(e.x), p1 = fast_exp2(e.y);
            pk[i] = pack_half2<kBf16>(p0, p1);
            sum2 = f2_add(sum2, f2_make(p0, p1));
            // O is normalised by the sum of the rounded weights it was built
            // from, so O / l is a weighted mean with consistent weights
            add_half2_to_f32<kBf16>(sr[2 * (i & 3)], sr[2 * (i & 3) + 1], pk[i]);
          }
          tmem_st16(pcol + col, pk);
        };
        // P(j) for keys [64*half, 64*half+64) goes to its columns [32*half, 32*half+32)
        pack_chunk(r0, half * 32);
        pack_chunk(r1, half * 32 + 16);
        const float2 sv = f2_split(sum2);
        l_run += sv.x + sv.y;
        lr_run += ((sr[0] + sr[1]) + (sr[2] + sr[3])) + ((sr[4] + sr[5]) + (sr[6] + sr[7]));

        if (j > 0 && __any_sync(0xffffffffu, raise)) {
          // the previous PV must be complete before O is rescaled.  The PV before
          // it, on the same barrier, was waited for above one tile ago, so this
          // wait is never more than one phase behind, and tiles that need no
          // rescale need not wait.
          if (!pf_wait_outlined(&bar_o[(gj - 1) & 1], (uint32_t)(((gj - 1) >> 1) & 1), &abort_flag, 7)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll 1
          for (int cc = 0; cc < HD / 32; ++cc) {
            uint32_t o[32];
            const uint32_t oa = lane_addr + C::O_COL + half * HD + cc * 32;
            tmem_ld32(oa, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(oa, o);
          }
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&bar_p[buf]);
      }
      if (ok && n > 0) {
        // the item's last P.V (the earlier ones are done or finish before it)
        ok = pf_wait_outlined(&bar_o[(gj - 1) & 1], (uint32_t)(((gj - 1) >> 1) & 1), &abort_flag, 8);
        tc_fence_after_sync();
      }
      // the row's sums are split over the two halves (one exchange buffer per
      // item parity: a half cannot get two epilogues ahead of its partner)
      const int ep = n_ep & 1;
      xch_l[ep][half][row] = l_run;
      xch_lr[ep][half][row] = lr_run;
      mbar_arrive(&bar_xe[wq]);
      if (ok) ok = pf_wait_outlined(&bar_xe[wq], (uint32_t)ep, &abort_flag, 10);
      ++n_ep;
      l_run += xch_l[ep][half ^ 1][row];
      lr_run += xch_lr[ep][half ^ 1][row];
      if (ok) {
        const bool row_valid = q_row < q_hi;
        const size_t row_idx = ((size_t)b * p.S_q + q_row) * p.h_q + h;
        const size_t lse_idx = ((size_t)b * p.h_q + h) * p.S_q + q_row;
        constexpr float kLn2 = 0.693147180559945309f;
        if constexpr (kMode != kModePartial) {
          const float inv_l = lr_run > 0.f ? 1.f / lr_run : 0.f;
          uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + row_idx * D + half * HD;
          const bool o_v8 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
#pragma unroll 1
          for (int cc = 0; cc < HD / 32; ++cc) {
            uint32_t o[32];
            if (n > 0) {
              tmem_ld32(lane_addr + C::O_COL + half * HD + cc * 32, o);
              tmem_ld_wait(o);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = 0u;
            }
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[i] = pack_half2<kBf16>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
            if (row_valid) {
              // a warp's store touches 32 rows: 32-byte pieces halve the requests
              // of 16-byte ones (the output's base decides)
              if (o_v8) {
                st_global_v8(orow + cc * 32, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
                st_global_v8(orow + cc * 32 + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
              } else {
                uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                  dst[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
              }
            }
          }
          if (p.lse != nullptr && row_valid && half == 0)
            p.lse[lse_idx] = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -CUDART_INF_F;
        } else {
          const bool any = l_run > 0.f && m_max != -CUDART_INF_F;
          const float f = any ? fast_exp2(m_run - m_max) : 0.f;  // re-reference to the true max
          // O re-weighted so that O / l equals the consistently normalised O_acc / lr
          const float fo = any ? f * (l_run / lr_run) : 0.f;
          float* orow = p.o_part + row_idx * D + half * HD;
#pragma unroll 1
          for (int cc = 0; cc < HD / 32; ++cc) {
            uint32_t o[32];
            if (n > 0) {
              tmem_ld32(lane_addr + C::O_COL + half * HD + cc * 32, o);
              tmem_ld_wait(o);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = 0u;
            }
            if (row_valid) {
              float4* dst = reinterpret_cast<float4*>(orow + cc * 32);
#pragma unroll
              for (int v4 = 0; v4 < 8; ++v4)
                dst[v4] = make_float4(__uint_as_float(o[4 * v4]) * fo, __uint_as_float(o[4 * v4 + 1]) * fo,
                                      __uint_as_float(o[4 * v4 + 2]) * fo, __uint_as_float(o[4 * v4 + 3]) * fo);
            }
          }
          if (row_valid && half == 0) {
            p.m_out[lse_idx] = any ? m_max * kLn2 : -CUDART_INF_F;
            p.l_out[lse_idx] = any ? l_run * f : 0.f;
          }
        }
      }
    }  // items
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool kBf16, int kMode, bool kOneChunk>
attn_status_t launch_prefill_variant(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                     const CUtensorMap& mv, dim3 grid, cudaStream_t s) {
  using C = PrefillCfg<D>;
  auto kern = prefill_kernel<D, kBf16, kMode, kOneChunk>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
    return ATTN_ERR_CUDA;
  kern<<<grid, C::THREADS, C::SMEM_BYTES, s>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Dense and window launches with one chunk, and every partial and jagged
// launch (always one KV range), take the single-chunk instantiations.
template <int D, bool kBf16>
attn_status_t launch_prefill_typed(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                   const CUtensorMap& mv, int mode, dim3 grid, cudaStream_t s) {
  const bool one = p.num_chunks == 1;
  switch (mode) {
    case kModeDense:
      return one ? launch_prefill_variant<D, kBf16, kModeDense, true>(p, mq, mk, mv, grid, s)
                 : launch_prefill_variant<D, kBf16, kModeDense, false>(p, mq, mk, mv, grid, s);
    case kModeWindow:
      return one ? launch_prefill_variant<D, kBf16, kModeWindow, true>(p, mq, mk, mv, grid, s)
                 : launch_prefill_variant<D, kBf16, kModeWindow, false>(p, mq, mk, mv, grid, s);
    case kModePartial:
      return one ? launch_prefill_variant<D, kBf16, kModePartial, true>(p, mq, mk, mv, grid, s) : ATTN_ERR_INVALID_ARG;
    case kModeJagged:
      return one ? launch_prefill_variant<D, kBf16, kModeJagged, true>(p, mq, mk, mv, grid, s) : ATTN_ERR_INVALID_ARG;
  }
  return ATTN_ERR_INVALID_ARG;
}

template <int D>
attn_status_t launch_prefill_dispatch(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                      const CUtensorMap& mv, int mode, bool bf16, dim3 grid, cudaStream_t s) {
  return bf16 ? launch_prefill_typed<D, true>(p, mq, mk, mv, mode, grid, s)
              : launch_prefill_typed<D, false>(p, mq, mk, mv, mode, grid, s);
}

}  // namespace attn
