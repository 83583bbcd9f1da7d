// Blockwise online-softmax attention forward on CTA pairs (head dimension 256;
// the template also takes 128): tcgen05 with cta_group::2, 256 query rows per
// pair sharing every K/V tile.
//
// What it computes, by source (the same as the paired kernel of head dims 64/128):
//  * "kernbench2 _gqa_prefill_long.py", gqa_prefill_long_kernel: per KV block,
//    scores = Q.K^T, m = rowmax, exp(scores - m), l = rowsum, O = exp . V,
//    merged into the running (m, l, O) with m_new = max(m, m_step) and the
//    factors exp(m - m_new), exp(m_step - m_new); O / l at the end.  The blocks
//    are 128-key tiles of a ring-order walk over the chunks.
//  * "[pallas] Support dependent Tile.end bounds in Pallas": the walk ends at
//    min(kv_end, tile_q.end); only the diagonal and tail tiles are masked.
//  * The module docstring of the prefill page, P6c: the query rows of one unit
//    are tiled over its processing elements, which share the unit's K/V.  Here
//    the unit is the two SMs of a TPC.
//
// Why pairs.  A single CTA computing a 128 x 128 x 256 score tile and its P.V
// moves 320 KB through its shared memory per KV tile (the S MMAs read 128 KB
// of Q and K, the P.V MMAs 64 KB of V, the copies write 128 KB) against 2048
// tensor cycles, more than the shared memory delivers in that time (128 B per
// cycle).  In a pair, one MMA instruction covers M = 256 rows: each CTA
// supplies its own 128 rows of Q (and of P, from its TMEM) and half of the B
// operand (64 keys of K; D / 2 columns of V, so one P.V MMA of N = D covers
// all of O), and each CTA's TMEM receives its own rows of S and O.  Per CTA
// and KV tile the shared memory then moves 192 KB: the S MMAs read 96 KB, the
// P.V MMAs 32 KB, the copies write 64 KB.
//
// Work: a pair item is 256 query rows that walk one KV sequence: two
// consecutive 128-row Q tiles of one (batch, head), the even CTA of the pair
// (rank 0) taking the first, walking the later tile's KV tiles (the earlier
// tile's rows see every key of all but the last tile, whose keys they mask);
// with GQA and an even group size, the same Q tile of two query heads of one
// KV group (identical walks).  Dense, partial and window launches are
// persistent: cluster c takes units c, c + clusters, ..., a unit being two
// items of one (batch, head or head pair) whose causal walks add up to the
// same length (items x and n - 1 - x), the longer first.  A jagged cluster
// takes one worklist item of 256 rows (in a causal sequence with an odd number
// of 128-row Q tiles, item t holds tiles 2t - 1 and 2t, item 0 tile 0 alone).
//
// CTA layout (480 threads; both CTAs of the pair run the same roles except
// where noted):
//   warp 0      TMA producer: this CTA's Q tile, then its halves of the K and V
//               tiles through a K ring and a V ring of shared-memory stages.
//               The copies of both CTAs complete on rank 0's barriers
//               (cta_group::2 form), which rank 0 arms for the bytes of both,
//               so one wait tells an issuer that both halves have landed.
//   warp 1      TMEM owner; rank 0: S issuer, S(j) = Q.K_j^T for the pair,
//               once K(j) has landed and both CTAs' softmax warps have read
//               S(j-1) (one barrier: the K stage's).
//   warp 10     rank 0: P.V issuer, once V(j) has landed and P(j) is written
//               (one barrier: the V stage's).  rank 1: idle.
//   warps 2..9  softmax of this CTA's 128 rows, two warps per row (a half of
//               the tile's keys and of O's columns each, the pair of warps
//               exchanging row maxima once per tile); their "S read" and "P
//               written" signals go to rank 0's K and V stage barriers (one
//               arrival per warp).
//               At the end of an item they leave each row's (m, l) in shared
//               memory and go on to the next item.
//   warps 11..14 epilogue of this CTA's 128 rows, one warp per TMEM lane
//               quarter: once the item's last P.V is done they read O out of
//               TMEM, signal "O free" to rank 0 (the next item's first P.V
//               waits for it) and store O / l and the LSE.
// Every MMA commit is multicast to both CTAs' barriers.  Every wait is bounded:
// a timeout sets the library's device status, the CTA skips its remaining
// work, waits for its copies in flight (a fixed time far longer than a copy
// takes: a stage's phase also counts softmax signals an aborted pipeline may
// never send, and rank 1's copies complete on rank 0's barriers) and (rank 0)
// for its MMAs, and both CTAs meet at a bounded exit handshake before freeing
// TMEM, so neither leaves while the other may still signal it.
#pragma once

#include <math_constants.h>

#include "prefill_common.cuh"

namespace attn {

template <int D_>
struct Cta2Cfg {
  static constexpr int D = D_;
  static constexpr int BM = 128;                // query rows per CTA (256 per pair)
  static constexpr int BN = 128;                // keys per KV tile
  static constexpr int KH = BN / 2;             // keys of a K tile each CTA holds
  static constexpr int VB = D / 128;            // 64-column blocks of V each CTA holds (its half of D)
  static constexpr int Q_BLOCK = 128 * 128;     // Q: 128 rows x 64 columns (128 B, swizzled)
  static constexpr int K_BLOCK = KH * 128;      // K half: 64 keys x 64 columns
  static constexpr int V_BLOCK = BN * 128;      // V: 128 keys x 64 columns
  static constexpr int Q_BYTES = BM * D * 2;    // 64 KB at head dim 256
  // one stage per K or V tile: this CTA's 64 keys x D columns of K, or the
  // tile's 128 keys x this CTA's D / 2 columns of V (rank r holds columns
  // [r D / 2, (r + 1) D / 2), so one P.V MMA of N = D covers all of O: at head
  // dim 256, 8 MMAs of 128 cycles per tile instead of 16 of 64, which halves
  // what the issuing thread must keep up with).  One barrier per tile: each wait of an MMA issuer
  // costs the tensor pipe a bubble (the wait holds the issuing thread until its
  // MMAs drain), and with one wait per slab (two per tile) the kernel ran
  // 1428-1510 vs 1471-1558 TFLOP/s on dense causal B=8 H=32 S=4096.
  static constexpr int STAGE_BYTES = KH * D * 2;
  // stages per ring (K tiles; V tiles): as many as fit next to Q and the static
  // part (2 at head dim 256, 5 at 128)
  static constexpr int RING = (213 * 1024 - Q_BYTES) / (2 * STAGE_BYTES);
  static constexpr int NST = 2 * RING;
  static constexpr int SMEM_BYTES = Q_BYTES + NST * STAGE_BYTES + 1024;  // + 1 KB alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  // TMEM (each CTA, its own 128 rows): S(j) in [0, 128); P(j) (16-bit) in
  // [P_COL + 64 (j % 2), +64); O in [O_COL, O_COL + 256)
  static constexpr uint32_t P_COL = 128;
  static constexpr uint32_t O_COL = 256;
  // softmax warps per query row: 2 (64 keys and 128 O columns each); 4 measured
  // slower (1364 vs 1428 TFLOP/s on dense causal B=8 H=32 S=4096)
  static constexpr int WPR = 2;
  static constexpr int SM_WARPS = 4 * WPR;      // softmax warps: WPR per TMEM lane quarter
  static constexpr int KW = BN / WPR;           // keys of a tile per softmax warp
  static constexpr int OW = D / WPR;            // O columns per softmax warp
  static constexpr int PV_WARP = 2 + SM_WARPS;  // the P.V issuer's warp (rank 0)
  static constexpr int EPI_WARP = 3 + SM_WARPS;  // first of the four epilogue warps
  static constexpr int THREADS = 32 * (EPI_WARP + 4);
  // 15 warps put four on three of the four SM sub-partitions (16K registers
  // each), so at most 128 registers per thread
  static constexpr int MAX_THREADS = 512;
  static constexpr uint16_t kBoth = 3;          // multicast mask of a commit: both CTAs
  static constexpr uint64_t kPeerCopyDrainNs = 200000;  // rank 1's wait for its copies after an abort
  static constexpr uint32_t kSignals = 2 * SM_WARPS;  // arrivals per phase: every softmax warp of the pair
  static constexpr uint32_t kEpiSignals = 2 * 4;       // "O free": every epilogue warp of the pair
  static_assert(WPR == 2 || WPR == 4, "softmax warps per row");
  static_assert(D == 128 || D == 256, "CTA-pair kernel: head dim 128 or 256");
  static_assert(BN * 64 * VB * 2 == STAGE_BYTES, "a K and a V stage are the same size");
  static_assert(RING >= 2, "K(j+1) must be loadable while K(j) is read");
  static_assert(O_COL + D <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES + 13 * 1024 <= 227 * 1024, "shared memory budget (static part < 13 KB)");
};

template <int D, bool kBf16, int kMode, bool kOneChunk>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cta2Cfg<D>::MAX_THREADS, 1)
    prefill_cta2_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                        const __grid_constant__ CUtensorMap mv, const PrefillParams p) {
  using C = Cta2Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_q, bar_qe, bar_fin, bar_exit;
  __shared__ uint64_t bar_o[2];  // PV(j) completes a phase of bar_o[j % 2] (both CTAs)
  __shared__ uint64_t bar_full[C::NST], bar_empty[C::NST];
  __shared__ uint64_t bar_s[2];
  __shared__ uint32_t tmem_slot;
  __shared__ uint32_t abort_flag;
  __shared__ float xch_max[2][C::WPR][128];  // [tile parity][key part][row]
  __shared__ uint64_t bar_x[2][4];  // exchange of a row's warps: [tile parity][lane quarter]
  // a finished item's row state, from the softmax warps to the epilogue warps:
  // [item parity][row] and [item parity][key part][row]
  __shared__ float ep_m[2][128], ep_mmax[2][128];
  __shared__ float ep_l[2][C::WPR][128], ep_lr[2][C::WPR][128];
  __shared__ uint64_t bar_ep_full[2], bar_ep_empty[2];  // [item parity]
  __shared__ uint64_t bar_ofree;  // rank 0: the epilogue warps of both CTAs have read O

  const uint32_t rank = cluster_ctarank();  // 0 issues the MMAs of the pair
  const int cl = (int)(blockIdx.x >> 1);
  const int n_cl = (int)(gridDim.x >> 1);

  // ------------------------------------------------------------ work items
  struct Item {
    int b, h;      // this CTA's batch and query head
    int q_lo, q_hi;  // this CTA's rows (none when q_hi <= q_lo)
    int u_lo, u_hi;  // the pair's rows: the walk's query range
    int kv_lo, kv_hi, q_pos0, kv_pos0;
    bool valid;
  };
  const int n_qt = (p.S_q + C::BM - 1) / C::BM;
  const int n_it = p.pair_heads ? n_qt : (n_qt + 1) / 2;  // items per (batch, head pair or head)
  const int n_ux = (n_it + 1) / 2;                        // units per (batch, head pair or head)
  const int n_y = p.pair_heads ? p.h_q / 2 : p.h_q;
  int n_my = 1;  // item slots of this pair
  if constexpr (kMode == kModeJagged) {
    if (cl >= *p.work_count) return;  // both CTAs of the pair read the same count
  } else {
    const long long units = (long long)n_ux * n_y * p.B;
    n_my = 2 * (int)((units - (long long)cl + n_cl - 1) / n_cl);
  }
  auto get_item = [&](int i) -> Item {
    Item it;
    it.valid = true;
    if constexpr (kMode == kModeJagged) {
      (void)i;
      // 256 rows of one sequence (cl < the item count: see the early return above)
      const int4 w = check_index(cl, *p.work_count, &g_prefill_status) ? p.work_items[cl] : make_int4(0, 0, 0, 0);
      it.b = 0;
      it.h = blockIdx.y;
      it.u_lo = w.z;
      it.u_hi = w.z + w.w;
      if (p.causal && (((w.y + C::BM - 1) / C::BM) & 1)) {
        // a causal sequence of an odd number of 128-row Q tiles: its first
        // tile (a one-tile walk) goes without a partner rather than its last
        // (the longest walk), so item t holds Q tiles 2t - 1 and 2t
        const int t = (w.z - w.x) / (2 * C::BM);
        it.u_lo = t == 0 ? w.x : w.x + (2 * t - 1) * C::BM;
        it.u_hi = min(it.u_lo + (t == 0 ? 1 : 2) * C::BM, w.x + w.y);
      }
      it.kv_lo = w.x;
      it.kv_hi = w.x + w.y;  // seq_offsets[seq_idx + 1]
      it.q_pos0 = 0;
      it.kv_pos0 = 0;
      it.q_lo = it.u_lo + C::BM * (int)rank;
      it.q_hi = min(it.q_lo + C::BM, it.u_hi);
    } else {
      const long long u = (long long)cl + (long long)(i >> 1) * n_cl;
      const int x = (int)(u % n_ux);
      const long long yb = u / n_ux;
      int xi;
      if (p.causal) {
        const int x_first = n_it - 1 - x;
        xi = (i & 1) ? x : x_first;
        it.valid = !(i & 1) || x < x_first;
      } else {
        xi = 2 * x + (i & 1);
        it.valid = xi < n_it;
      }
      it.b = (int)(yb / n_y);
      const int y = (int)(yb % n_y);
      if (p.pair_heads) {
        it.h = 2 * y + (int)rank;
        it.u_lo = xi * C::BM;
        it.u_hi = min(it.u_lo + C::BM, p.S_q);
        it.q_lo = it.u_lo;
        it.q_hi = it.u_hi;
      } else {
        it.h = y;
        it.u_lo = xi * 2 * C::BM;
        it.u_hi = min(it.u_lo + 2 * C::BM, p.S_q);
        it.q_lo = it.u_lo + C::BM * (int)rank;
        it.q_hi = min(it.q_lo + C::BM, it.u_hi);
      }
      it.kv_lo = p.kv_lo;
      it.kv_hi = p.kv_hi;
      it.q_pos0 = p.q_pos0;
      it.kv_pos0 = p.kv_pos0;
    }
    return it;
  };
  // the pair's walk: every role of both CTAs derives the same one
  auto item_walk = [&](const Item& it, TileWalk& w) -> int {
    w.init(it.u_lo, it.u_hi, it.kv_lo, it.kv_hi, it.q_pos0, it.kv_pos0, p.causal, kOneChunk ? 1 : p.num_chunks, C::BN,
           kMode == kModeWindow ? p.window : -1);
    return w.count();
  };

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
    mbar_init(&bar_fin, 2);  // one commit per MMA issuer, multicast to both CTAs
    mbar_init(&bar_exit, 1);
    // a K stage's fill for tile j completes once its copies have landed and
    // the pair's softmax warps have read S(j - 1) (the one S buffer is free);
    // a V stage's fill for tile j once its copies have landed and the softmax
    // warps have written P(j): one wait per tile for each MMA issuer
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&bar_full[s], 1 + C::kSignals);
      mbar_init(&bar_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_s[i], 1);
      for (int q4 = 0; q4 < 4; ++q4) mbar_init(&bar_x[i][q4], 32 * C::WPR);
      mbar_init(&bar_ep_full[i], 32 * C::SM_WARPS);
      mbar_init(&bar_ep_empty[i], 32 * 4);
    }
    mbar_init(&bar_ofree, C::kEpiSignals);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_cta2(&tmem_slot, C::TMEM_COLS);
    tmem_relinquish_cta2();
  }
  tc_fence_before_sync();
  __syncthreads();
  // both CTAs' barriers are initialised before either signals the other's
  cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    // ========================================================== TMA producer (both CTAs)
    if (lane == 0) {
      prefetch_tensormap(&mq);
      prefetch_tensormap(&mk);
      prefetch_tensormap(&mv);
      // a tile load whose coordinates fail the checked build's test loads tile
      // (0, 0, 0, 0) instead, so the pipeline's barriers still complete
      auto load = [&](void* dst, const CUtensorMap* map, uint32_t bar, int c0, int c1, int c2, int c3, int heads,
                      int rows) {
        if (!check_tile(c0, c1, c2, c3, D, heads, rows, p.B, 256, &g_prefill_status)) c0 = c1 = c2 = c3 = 0;
        tma_load_4d_pair(dst, map, bar, c0, c1, c2, c3);
      };
      int filled[2] = {0, 0};  // tiles issued into the K ring and the V ring
      int q_loads = 0;
      bool ok = true;
      int hk = 0, bb = 0;
      // fill f of a ring goes to its stage f % RING, once the pair's MMAs have
      // released fill f - RING of that stage (the commit reaches both CTAs).
      // Both CTAs' copies of a fill complete on rank 0's barrier, which rank 0
      // arms for the bytes of both.
      auto push_tile = [&](int ring, int kstart) -> bool {
        int& fills = filled[ring];
        const int stage = ring * C::RING + fills % C::RING;
        const uint32_t phase = (uint32_t)((fills / C::RING) & 1);
        if (!pf_wait_outlined(&bar_empty[stage], phase ^ 1u, &abort_flag, 1)) return false;
        uint8_t* dst = sKV + stage * C::STAGE_BYTES;
        if (rank == 0) mbar_arrive_expect_tx(&bar_full[stage], 2 * C::STAGE_BYTES);
        const uint32_t full0 = mapa_shared(&bar_full[stage], 0);
        if (ring == 0) {
          // K: this CTA's 64 keys of the tile, all 256 columns
          for (int blk = 0; blk < D / 64; ++blk)
            load(dst + blk * C::K_BLOCK, &mk, full0, blk * 64, hk, kstart + C::KH * (int)rank, bb, p.h_kv, p.S_kv);
        } else {
          // V: the tile's 128 keys, this CTA's 64 columns of each 128-column half
          for (int vb = 0; vb < C::VB; ++vb)
            load(dst + vb * C::V_BLOCK, &mv, full0, (int)rank * (D / 2) + 64 * vb, hk, kstart, bb, p.h_kv, p.S_kv);
        }
        ++fills;
        return true;
      };
      for (int i = 0; ok && i < n_my; ++i) {
        const Item it = get_item(i);
        if (!it.valid) continue;
        TileWalk walk;
        const int n = item_walk(it, walk);
        if (n == 0) continue;
        hk = it.h / p.group;
        bb = it.b;
        // the Q buffer is free once the previous item's S MMAs are done
        if (q_loads > 0 && !pf_wait_outlined(&bar_qe, (uint32_t)((q_loads - 1) & 1), &abort_flag, 13)) {
          ok = false;
          break;
        }
        if (rank == 0) mbar_arrive_expect_tx(&bar_q, 2 * C::Q_BYTES);
        const uint32_t q0 = mapa_shared(&bar_q, 0);
        for (int blk = 0; blk < D / 64; ++blk)
          load(sQ + blk * C::Q_BLOCK, &mq, q0, blk * 64, it.h, it.q_lo, it.b, p.h_q, p.S_q);
        ++q_loads;
        TileWalk kw = walk, vw = walk;
        int ch, st, me;
        kw.next(ch, st, me);
        ok = push_tile(0, st);
        for (int j = 0; ok && j < n; ++j) {
          if (j + 1 < n) {
            kw.next(ch, st, me);
            ok = push_tile(0, st);
            if (!ok) break;
          }
          vw.next(ch, st, me);
          ok = push_tile(1, st);
        }
      }
      if (abort_flag) {
        // copies may still be landing in this CTA's shared memory: wait for
        // them.  A stage's phase also counts softmax signals that an aborted
        // pipeline may never send, and rank 1's copies complete on rank 0's
        // barriers, which it cannot poll, so both CTAs wait a fixed time far
        // longer than a copy takes (the CTAs then meet at the exit handshake,
        // so rank 0's barriers outlive rank 1's copies); rank 0 first drains
        // its Q barrier, which counts copies only.
        if (rank == 0 && q_loads > 0) pf_drain(&bar_q, (uint32_t)((q_loads - 1) & 1));
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < C::kPeerCopyDrainNs) {
        }
      }
    }
  } else if (warp == 1 && rank != 0) {
    // ========================================================== rank 1, warp 1
    // rank 0's MMAs read this CTA's shared memory and write its TMEM: they
    // finish before this CTA tears down (the final commits reach both CTAs)
    if (lane == 0) pf_drain(&bar_fin, 0);
  } else if (warp == 1 || warp == C::PV_WARP) {
    // ========================================================== MMA issuers (rank 0)
    // Warp 1 issues S(j), warp PV_WARP PV(j), for the whole pair.  Each only
    // waits on work of other roles, twice per tile (a wait stalls until the
    // thread's own issued tcgen05 work has drained, a bubble in the tensor
    // pipe): the S issuer on the softmax having read S(j-1) and on K(j), the PV
    // issuer on P(j) and on V(j).
    if (lane == 0 && rank == 0) {
      constexpr uint32_t kIdescS = idesc_f16_f32acc(256, C::BN, kBf16, false);
      constexpr uint32_t kIdescPV = idesc_f16_f32acc(256, D, kBf16, true);
      const uint32_t skv = smem_u32(sKV);
      auto wait_tile = [&](int ring, int f, uint32_t site) -> bool {
        const int stage = ring * C::RING + f % C::RING;
        const uint32_t ph = (uint32_t)((f / C::RING) & 1);
        if (!pf_wait_outlined(&bar_full[stage], ph, &abort_flag, site)) return false;
        tc_fence_after_sync();
        return true;
      };
      bool ok = true;
      int g = 0;          // S (or PV) groups issued so far, all items: barrier phases
      int tile_base = 0;  // tiles of this issuer's ring taken by the earlier items
      int q_used = 0;     // Q tiles consumed (S issuer)
      int o_items = 0;    // items whose P.V MMAs were issued (P.V issuer)
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
            {
              // K(j) has landed and the softmax warps of both CTAs have read
              // S(j-1): the one S buffer is free
              const int tl = tile_base + j;
              ok = wait_tile(0, tl, 2);
              if (!ok) break;
              const uint64_t kdesc = smem_desc_sw128(skv + (tl % C::RING) * C::STAGE_BYTES, 16, 1024);
#pragma unroll
              for (int ks = 0; ks < D / 16; ++ks) {
                // 16 columns of D per MMA: 32 bytes inside a 128-byte swizzle row,
                // the next 64-column block every four steps
                const uint32_t qoff = (ks / 4) * C::Q_BLOCK + (ks % 4) * 32;
                const uint32_t koff = (ks / 4) * C::K_BLOCK + (ks % 4) * 32;
                mma_ss_cta2(tmem, desc_advance(qdesc, qoff), desc_advance(kdesc, koff), kIdescS, ks != 0);
              }
              mma_commit_cta2(&bar_empty[tl % C::RING], C::kBoth);
            }
            if (!ok) break;
            mma_commit_cta2(&bar_s[g & 1], C::kBoth);
          }
          // the item's S MMAs, the last readers of its Q, release both Q buffers
          if (ok) mma_commit_cta2(&bar_qe, C::kBoth);
        } else {
          // the item's first P.V starts O afresh: the epilogue warps of both CTAs
          // have read the previous item's O out of TMEM
          if (o_items > 0) {
            ok = pf_wait_outlined(&bar_ofree, (uint32_t)((o_items - 1) & 1), &abort_flag, 14);
            if (!ok) break;
            tc_fence_after_sync();
          }
          ++o_items;
          for (int j = 0; ok && j < n; ++j, ++g) {
            // V(j) has landed and P(j) of both CTAs is in TMEM (one barrier)
            const uint32_t p_tmem = tmem + C::P_COL + static_cast<uint32_t>((g & 1) * 64);
            const uint32_t acc0 = j > 0 ? 1u : 0u;  // the item's first PV starts O afresh
            {
              const int tl = tile_base + j;
              ok = wait_tile(1, tl, 4);
              if (!ok) break;
              const int stage = C::RING + tl % C::RING;
              {
                // this CTA's D / 2 columns of V: 64-column blocks 16 KB apart
                const uint64_t vdesc = smem_desc_sw128(skv + stage * C::STAGE_BYTES, C::V_BLOCK, 1024);
                // 16 keys of V per MMA (16 rows of 128 bytes in each block)
#pragma unroll
                for (int ks = 0; ks < C::BN / 16; ++ks)
                  mma_ts_cta2(tmem + C::O_COL, p_tmem + ks * 8, desc_advance(vdesc, ks * 2048), kIdescPV,
                              ks > 0 ? 1u : acc0);
              }
              mma_commit_cta2(&bar_empty[stage], C::kBoth);
            }
            if (!ok) break;
            mma_commit_cta2(&bar_o[g & 1], C::kBoth);
          }
        }
        tile_base += n;
      }
      // every MMA either issuer issued must finish before TMEM is released (both CTAs)
      mma_commit_cta2(&bar_fin, C::kBoth);
      pf_drain(&bar_fin, 0);
    }
  } else if (warp >= 2 && warp < 2 + C::SM_WARPS) {
    // ========================================================== softmax (both CTAs)
    // WPR warps share each TMEM lane quarter: warp 2 + 4 kq + (wq - 2) mod 4 ...
    // takes key part kq of every row of lane quarter wq (keys [KW kq, KW kq + KW)
    // of a tile, O columns [OW kq, OW kq + OW)).  The row's warps exchange their
    // maxima once per tile through shared memory, so all take identical
    // decisions.
    constexpr int KW = C::KW, OW = C::OW, NKC = KW / 32;
    const int sw = warp - 2;        // 0 .. SM_WARPS - 1
    const int wq = warp & 3;        // TMEM lane quarter this warp may access
    const int kq = sw >> 2;         // key part of this warp
    const int row = wq * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float c = p.scale_log2;  // > 0
    // one arrival per warp on rank 0's barrier of a stage: local there,
    // remote from rank 1
    auto signal = [&](int stage) {
      if (rank == 0)
        mbar_arrive(&bar_full[stage]);
      else
        mbar_arrive_remote(mapa_shared(&bar_full[stage], 0));
    };
    // the K stage of the first tile waits for no S read
    __syncwarp();
    if (lane == 0) signal(0);
    bool ok = true;
    int gj = 0;    // tiles so far, all items: the phases of the per-tile barriers
    int n_ep = 0;  // epilogues so far
    for (int i = 0; ok && i < n_my; ++i) {
      const Item it = get_item(i);
      if (!it.valid) continue;
      TileWalk sw_walk;
      const int n = item_walk(it, sw_walk);
      const int q_lo = it.q_lo, q_hi = it.q_hi, q_pos0 = it.q_pos0, kv_pos0 = it.kv_pos0;
      const int q_row = q_lo + row;
      float m_run = -CUDART_INF_F;   // reference max (exp2 domain), raised lazily
      float l_run = 0.f;             // this part's sum of exp2(x - m_run) in fp32: l and LSE
      float lr_run = 0.f;            // this part's sum of the rounded P the MMA multiplies V by
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
        uint32_t r[NKC][32];
#pragma unroll
        for (int cc = 0; cc < NKC; ++cc) tmem_ld32(lane_addr + kq * KW + cc * 32, r[cc]);
#pragma unroll
        for (int cc = 0; cc < NKC; ++cc) tmem_ld_wait(r[cc]);
        // S(j) is in registers: the S issuer may overwrite the buffer with S(j+1)
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) signal((gj + 1) % C::RING);  // the K stage of tile gj + 1

        // mask the diagonal / tail tile (key kstart + i is visible iff i < lim)
        // and, under a sliding window, the tiles at its lower edge (iff i >= flo);
        // the pair's walk may hold tiles that none of this CTA's rows sees
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
          // limits within this part, clamped to its keys
          const int ilh = clamp_limit(lim - kq * KW, KW), ifh = clamp_limit(flo - kq * KW, KW);
          const uint32_t ninf = __float_as_uint(-CUDART_INF_F);
#pragma unroll
          for (int cc = 0; cc < NKC; ++cc) apply_mask(r[cc], chunk_mask(cc * 32, ifh, ilh), ninf);
        }
        float mx8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          mx8[k] = fmax3(__uint_as_float(r[0][k]), __uint_as_float(r[0][k + 8]), __uint_as_float(r[0][k + 16]));
          mx8[k] = fmaxf(mx8[k], __uint_as_float(r[0][k + 24]));
#pragma unroll
          for (int cc = 1; cc < NKC; ++cc) {
            mx8[k] = fmax3(mx8[k], __uint_as_float(r[cc][k]), __uint_as_float(r[cc][k + 8]));
            mx8[k] = fmax3(mx8[k], __uint_as_float(r[cc][k + 16]), __uint_as_float(r[cc][k + 24]));
          }
        }
        float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
        // the row's parts see each other's max
        xch_max[buf][kq][row] = mx;
        mbar_arrive(&bar_x[buf][wq]);
        if (!pf_wait_outlined(&bar_x[buf][wq], (uint32_t)((gj >> 1) & 1), &abort_flag, 9)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int o = 1; o < C::WPR; ++o) mx = fmaxf(mx, xch_max[buf][(kq + o) % C::WPR][row]);
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
        // P(j) for keys [KW kq, KW kq + KW) goes to its columns [KW / 2 kq, +KW / 2)
#pragma unroll
        for (int cc = 0; cc < NKC; ++cc) {
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 e = f2_split(f2_fma(f2_make_u(r[cc][2 * k], r[cc][2 * k + 1]), c2, nm2));
            const float p0 = fast_exp2(e.x), p1 = fast_exp2(e.y);
            pk[k] = pack_half2<kBf16>(p0, p1);
            sum2 = f2_add(sum2, f2_make(p0, p1));
            // O is normalised by the sum of the rounded weights it was built
            // from, so O / l is a weighted mean with consistent weights
            add_half2_to_f32<kBf16>(sr[2 * (k & 3)], sr[2 * (k & 3) + 1], pk[k]);
          }
          tmem_st16(pcol + kq * (KW / 2) + cc * 16, pk);
        }
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
          for (int cc = 0; cc < OW / 32; ++cc) {
            uint32_t o[32];
            const uint32_t oa = lane_addr + C::O_COL + kq * OW + cc * 32;
            tmem_ld32(oa, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            tmem_st32(oa, o);
          }
        }
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) signal(C::RING + gj % C::RING);  // the V stage of tile gj
      }
      if (ok && n > 0) {
        // hand the row's state to the epilogue warps (one buffer per item
        // parity: before a buffer is reused, the epilogue warps have read what
        // the item two back left in it)
        const int eb = n_ep & 1;
        if (n_ep >= 2) ok = pf_wait_outlined(&bar_ep_empty[eb], (uint32_t)(((n_ep >> 1) - 1) & 1), &abort_flag, 15);
        if (ok) {
          ep_l[eb][kq][row] = l_run;
          ep_lr[eb][kq][row] = lr_run;
          if (kq == 0) {
            ep_m[eb][row] = m_run;
            ep_mmax[eb][row] = m_max;
          }
          mbar_arrive(&bar_ep_full[eb]);
        }
        ++n_ep;
      }
    }  // items
  } else if (warp >= C::EPI_WARP) {
    // ========================================================== epilogue (both CTAs)
    // One warp per TMEM lane quarter (warp w takes the rows of quarter w mod 4,
    // one row per thread).  Per item with tiles: the row's state from the
    // softmax warps, then, once the item's last P.V is done, O out of TMEM,
    // after which the P.V issuer may start the next item's O while these warps
    // normalise and store this one.  The softmax warps meanwhile already work
    // on the next item, so an item boundary costs them no epilogue.
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t ofree_remote = mapa_shared(&bar_ofree, 0);
    const bool o_v8 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
    constexpr float kLn2 = 0.693147180559945309f;
    bool ok = true;
    int gj = 0;    // tiles so far, all items
    int n_ep = 0;  // items with tiles so far
    for (int i = 0; ok && i < n_my; ++i) {
      const Item it = get_item(i);
      if (!it.valid) continue;
      TileWalk ep_walk;
      const int n = item_walk(it, ep_walk);
      float m_run = -CUDART_INF_F, l_run = 0.f, lr_run = 0.f, m_max = -CUDART_INF_F;
      if (n > 0) {
        const int eb = n_ep & 1;
        if (!pf_wait_outlined(&bar_ep_full[eb], (uint32_t)((n_ep >> 1) & 1), &abort_flag, 16)) {
          ok = false;
          break;
        }
        m_run = ep_m[eb][row];
        m_max = ep_mmax[eb][row];
#pragma unroll
        for (int o = 0; o < C::WPR; ++o) {
          l_run += ep_l[eb][o][row];
          lr_run += ep_lr[eb][o][row];
        }
        mbar_arrive(&bar_ep_empty[eb]);
        ++n_ep;
        gj += n;
        // the item's last P.V (the earlier ones finish before it)
        if (!pf_wait_outlined(&bar_o[(gj - 1) & 1], (uint32_t)(((gj - 1) >> 1) & 1), &abort_flag, 8)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
      }
      const int q_row = it.q_lo + row;
      const size_t row_idx = ((size_t)it.b * p.S_q + q_row) * p.h_q + it.h;
      const size_t lse_idx = ((size_t)it.b * p.h_q + it.h) * p.S_q + q_row;
      const long long rows_all = (long long)p.B * p.S_q * p.h_q;
      const bool row_valid = q_row < it.q_hi && check_index((long long)row_idx, rows_all, &g_prefill_status) &&
                             check_index((long long)lse_idx, rows_all, &g_prefill_status);
      // O / lr in the input type; a partial's fp32 O re-referenced to the true
      // max and re-weighted so that O / l equals the consistently normalised
      // O_acc / lr
      const bool any = l_run > 0.f && m_max != -CUDART_INF_F;
      const float f = any ? fast_exp2(m_run - m_max) : 0.f;
      float so;
      if constexpr (kMode != kModePartial)
        so = lr_run > 0.f ? 1.f / lr_run : 0.f;
      else
        so = any ? f * (l_run / lr_run) : 0.f;
      auto emit = [&](int cc, const uint32_t(&o)[32]) {
        if (!row_valid) return;
        if constexpr (kMode != kModePartial) {
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            w[k] = pack_half2<kBf16>(__uint_as_float(o[2 * k]) * so, __uint_as_float(o[2 * k + 1]) * so);
          uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + row_idx * D + cc * 32;
          // a warp's store touches 32 rows: 32-byte pieces halve the requests
          // of 16-byte ones (the output's base decides)
          if (o_v8) {
            st_global_v8(orow, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
            st_global_v8(orow + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) dst[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(p.o_part + row_idx * D + cc * 32);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            dst[v4] = make_float4(__uint_as_float(o[4 * v4]) * so, __uint_as_float(o[4 * v4 + 1]) * so,
                                  __uint_as_float(o[4 * v4 + 2]) * so, __uint_as_float(o[4 * v4 + 3]) * so);
        }
      };
      if (n > 0) {
        // two chunks of 32 columns in flight: chunk c + 1 loads while chunk c
        // is normalised and stored
        uint32_t oa[32], ob[32];
        tmem_ld32(lane_addr + C::O_COL, oa);
        tmem_ld_wait(oa);
#pragma unroll 1
        for (int cc = 0; cc < D / 32; cc += 2) {
          tmem_ld32(lane_addr + C::O_COL + (cc + 1) * 32, ob);
          emit(cc, oa);
          tmem_ld_wait(ob);
          if (cc + 2 < D / 32) {
            tmem_ld32(lane_addr + C::O_COL + (cc + 2) * 32, oa);
          } else {
            // all of O is read: the next item's first P.V may overwrite it
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
              if (rank == 0)
                mbar_arrive(&bar_ofree);
              else
                mbar_arrive_remote(ofree_remote);
            }
          }
          emit(cc + 1, ob);
          if (cc + 2 < D / 32) tmem_ld_wait(oa);
        }
      } else {
        // no visible key: O = 0 (and LSE = -inf)
        uint32_t z[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) z[k] = 0u;
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) emit(cc, z);
      }
      if constexpr (kMode != kModePartial) {
        if (p.lse != nullptr && row_valid) p.lse[lse_idx] = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -CUDART_INF_F;
      } else if (row_valid) {
        p.m_out[lse_idx] = any ? m_max * kLn2 : -CUDART_INF_F;
        p.l_out[lse_idx] = any ? l_run * f : 0.f;
      }
    }  // items
  }

  // ------------------------------------------------------------ teardown
  // Every thread of this CTA is done with TMEM and with signalling the other
  // CTA.  The two CTAs then meet (bounded): neither exits, nor frees the
  // pair's TMEM, while the other may still signal its barriers.
  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_remote(mapa_shared(&bar_exit, rank ^ 1u));
    pf_drain(&bar_exit, 0);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_cta2(tmem, C::TMEM_COLS);
  }
}

template <int D, bool kBf16, int kMode, bool kOneChunk>
attn_status_t launch_cta2_variant(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                  const CUtensorMap& mv, dim3 grid, cudaStream_t s) {
  using C = Cta2Cfg<D>;
  auto kern = prefill_cta2_kernel<D, kBf16, kMode, kOneChunk>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (grid.x == 0 || grid.x % 2 != 0) return ATTN_ERR_INVALID_ARG;
  kern<<<grid, C::THREADS, C::SMEM_BYTES, s>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Dense and window launches with one chunk, and every partial and jagged
// launch (always one KV range), take the single-chunk instantiations.
template <int D, bool kBf16>
attn_status_t launch_cta2_typed(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                const CUtensorMap& mv, int mode, dim3 grid, cudaStream_t s) {
  const bool one = p.num_chunks == 1;
  switch (mode) {
    case kModeDense:
      return one ? launch_cta2_variant<D, kBf16, kModeDense, true>(p, mq, mk, mv, grid, s)
                 : launch_cta2_variant<D, kBf16, kModeDense, false>(p, mq, mk, mv, grid, s);
    case kModeWindow:
      return one ? launch_cta2_variant<D, kBf16, kModeWindow, true>(p, mq, mk, mv, grid, s)
                 : launch_cta2_variant<D, kBf16, kModeWindow, false>(p, mq, mk, mv, grid, s);
    case kModePartial:
      return one ? launch_cta2_variant<D, kBf16, kModePartial, true>(p, mq, mk, mv, grid, s) : ATTN_ERR_INVALID_ARG;
    case kModeJagged:
      return one ? launch_cta2_variant<D, kBf16, kModeJagged, true>(p, mq, mk, mv, grid, s) : ATTN_ERR_INVALID_ARG;
  }
  return ATTN_ERR_INVALID_ARG;
}

template <int D>
attn_status_t launch_cta2_dispatch(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                          const CUtensorMap& mv, int mode, bool bf16, dim3 grid, cudaStream_t s) {
  return bf16 ? launch_cta2_typed<D, true>(p, mq, mk, mv, mode, grid, s)
              : launch_cta2_typed<D, false>(p, mq, mk, mv, mode, grid, s);
}

}  // namespace attn
