// Blockwise online-softmax attention forward for head dimensions 64 and 128:
// two 128-row Q sub-tiles per CTA that share every K/V tile.
//
// What it computes is the same as the head-dim-256 kernel (prefill_cta2_kernel.cuh):
// per KV tile, S = Q.K^T, the running (m, l, O) updated by online softmax
// ("kernbench2 _gqa_prefill_long.py", step 0 partial and the ring-step merge),
// O / l at the end, over the tiles of a ring-order walk that stops at
// min(kv_end, tile_q.end) ("[pallas] Support dependent Tile.end bounds in
// Pallas").  The difference is the amount of K/V traffic per FLOP: each K/V
// byte brought into shared memory feeds 256 query rows instead of 128, which
// halves what the TMA has to deliver per tensor-core cycle (one 128-row tile
// needs ~64 B/clk/SM at full MMA rate, about the measured TMA ceiling).
//
// Pairing: for GQA the sub-tiles are two query heads of one KV group at the
// same Q tile (identical tile walks); otherwise they are two consecutive Q
// tiles of one head / sequence and share the walk of the later one, the
// earlier sub-tile sitting out the tiles it cannot see (no masked-only work).
//
// A CTA walks a list of work items (a Q tile pair with its KV walk): the next
// item's Q and first K/V tiles load, and its first S tiles are computed, while
// the previous item's last P.V products and epilogue finish.  Jagged and
// sliding-window launches are persistent (one CTA per SM, items in a snake
// order over the CTAs, longest first), because their items are short (a
// window item walks about window / 128 tiles): persistence measured +2.6 % on
// the 4096-key window.  Dense launches run one item per CTA in the hardware's
// launch order, which keeps the CTAs that run at one time on the K/V of one
// head: on the long causal ring the persistent form measured -1.7 % (and an
// earlier static split 1.65x the DRAM reads of that order).
//
// CTA layout (352 threads):
//   warp 0      TMA producer: per item both Q sub-tiles (once the previous
//               item's MMAs are done with the Q buffer), then K(0), V(0),
//               K(1), V(1), ... through a ring of NST stages (one stage = one
//               K or V tile) that runs on across items.
//   warp 1      TMEM owner (512 columns: S_A, S_B, O_A, O_B) and S issuer:
//               S_A(j), S_B(j) per tile, each once its sub-tile's previous
//               P.V has read the P held in its S buffer.
//   warps 2..5  softmax + epilogue of sub-tile A, one query row per thread.
//   warps 6..9  the same for sub-tile B.
//   warp 10     P.V issuer: PV_A(j), PV_B(j) as each P becomes ready, so one
//               sub-tile's MMAs run while the other sub-tile's softmax runs.
// P(j) of a sub-tile (bf16/fp16) overwrites the first 64 columns of its S
// buffer and is the TMEM A operand of P.V.  Every wait is bounded.
#pragma once

#include <type_traits>

#include "prefill_common.cuh"

namespace attn {

template <int D>
struct PairCfg {
  static constexpr int BM = 128;
  static constexpr int BN = 128;
  static constexpr int BLOCK_BYTES = 128 * 128;  // one TMA block: 128 rows x 128 bytes
  static constexpr int Q_BYTES = BM * D * 2;     // one sub-tile
  static constexpr int SLAB_BYTES = BN * D * 2;  // one K or V tile
  static constexpr int NST = (224 * 1024 - 2 * Q_BYTES) / SLAB_BYTES;
  static constexpr int SMEM_BYTES = 2 * Q_BYTES + NST * SLAB_BYTES + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t O_COL = 256;  // S_A 0..127, S_B 128..255, O_A 256.., O_B 256+D..
  static constexpr int THREADS = 352;
  static_assert(D == 64 || D == 128, "paired kernel: head dim 64 or 128");
  static_assert(NST >= 3, "K(j+1) must be loadable while K(j) and V(j) are held");
  // One ring holds K and V.  The producer pushes, over all items, K0 V0 K1 V1
  // ... (each item pushes 2n slabs starting with K), so slab s is a K tile iff s
  // is even and lives in stage s % NST, round s / NST.  Before an issuer waits
  // for slab s, the stage's previous fill, slab s - NST, must be complete: a
  // parity wait cannot tell it from slab s (the phase before the awaited one
  // reads as complete).  With NST even, slab s - NST is of the same kind and
  // the same issuer waited for it earlier.  With NST odd (head dim 128: 5) it
  // belongs to the other issuer, and the order of the waits is what excludes
  // the hazard (see ORDER at the two wait sites); checked builds verify it at
  // run time.  Split K and V rings would exclude it structurally, but measured
  // 1.2 % (ring), 2.3-3.6 % (sliding window) and up to 2.2 % (jagged) slower
  // with either split of the five stages.
  static_assert(NST % 2 == 0 || NST >= 5, "the ordering argument for an odd ring needs five stages or more");
  static_assert(SMEM_BYTES <= 227 * 1024 - 512, "shared memory budget");
};

struct SubTile {
  int h, q_lo, q_hi;
  __device__ bool empty() const { return q_hi <= q_lo; }
};

// One work item of the paired kernel: two sub-tiles and the KV range they walk.
struct PairItem {
  int b, kv_lo, kv_hi, q_pos0, kv_pos0;
  SubTile st0, st1;
};

// Number of work units of a launch: jagged, (sequence, head) pairs from the
// device worklist's unit table; otherwise single items.
template <int kMode>
__device__ __forceinline__ int pair_item_count(const PrefillParams& p) {
  if constexpr (kMode == kModeJagged) return p.work_count[1] * p.h_q;
  return p.n_items;
}

// Work unit k: items [i0, i0 + n) of head h.  A jagged unit is every Q tile of
// one (sequence, head), first to last, taken back to back by one CTA so that
// each tile re-reads from L2 the K/V its predecessors brought in
// ("Grouping" in "[pallas] Support dependent Tile.end bounds in Pallas":
// successive Q work items reuse the resident K/V range).  The worklist's item
// count bounds the unit's items.
struct PairUnit {
  int i0, n, h;
};
template <int kMode>
__device__ __forceinline__ PairUnit pair_unit(const PrefillParams& p, int k) {
  if constexpr (kMode == kModeJagged) {
    const int2 u = check_index(k / p.h_q, p.work_count[1], &g_prefill_status) ? p.work_units[k / p.h_q] : make_int2(0, 0);
    const int n = min(u.y, *p.work_count - u.x);
    return PairUnit{u.x, n > 0 ? n : 0, k % p.h_q};
  } else {
    return PairUnit{k, 1, 0};
  }
}

// Item k of the launch (jagged: worklist item k for head h).  Dense / partial
// items: the Q tiles of one head (pair) and batch are consecutive, longest
// causal walk first, so the CTAs that run at one time share the K/V of one
// head in L2.
template <int kMode>
__device__ __forceinline__ PairItem pair_item(const PrefillParams& p, int k, int h) {
  constexpr int BM = 128;
  PairItem it;
  if constexpr (kMode == kModeJagged) {
    // a 256-row Q tile of one sequence (a failed check reads an empty item)
    const int4 w = check_index(k, *p.work_count, &g_prefill_status) ? p.work_items[k] : make_int4(0, 0, 0, 0);
    int lo = w.z, mid = w.z + min(w.w, BM), hi = w.z + w.w;
    if (p.causal) {
      // A causal sequence of an odd number m of 128-row Q tiles leaves one
      // tile without a partner.  Its first tile (a one-tile walk) takes that
      // place rather than its last (the longest walk): item t of the sequence
      // holds Q tiles 2t - 1 and 2t, item 0 tile 0 alone.  The item count,
      // ceil(m / 2), is the worklist's.
      const int m = (w.y + BM - 1) / BM;
      if (m & 1) {
        const int t = (w.z - w.x) / (2 * BM);
        const int seq_end = w.x + w.y;
        lo = t == 0 ? w.x : w.x + (2 * t - 1) * BM;
        mid = min(lo + BM, seq_end);
        hi = t == 0 ? mid : min(lo + 2 * BM, seq_end);
      }
    }
    it.b = 0;
    it.st0 = SubTile{h, lo, mid};
    it.st1 = SubTile{h, mid, hi};
    it.kv_lo = w.x;
    it.kv_hi = w.x + w.y;  // seq_offsets[seq_idx + 1]
    it.q_pos0 = 0;
    it.kv_pos0 = 0;
  } else {
    (void)h;
    const int yb = k / p.n_qt;
    const int t_rank = k - yb * p.n_qt;
    const int y = yb % p.n_y;
    it.b = yb / p.n_y;
    const int t = p.causal ? p.n_qt - 1 - t_rank : t_rank;
    it.kv_lo = p.kv_lo;
    it.kv_hi = p.kv_hi;
    it.q_pos0 = p.q_pos0;
    it.kv_pos0 = p.kv_pos0;
    if (p.pair_heads) {
      const int lo = t * BM, hi = min(lo + BM, p.S_q);
      it.st0 = SubTile{2 * y, lo, hi};
      it.st1 = SubTile{2 * y + 1, lo, hi};
    } else {
      const int lo = t * 2 * BM;
      const int mid = min(lo + BM, p.S_q), hi = min(lo + 2 * BM, p.S_q);
      it.st0 = SubTile{y, lo, mid};
      it.st1 = SubTile{y, mid, hi};
    }
  }
  return it;
}

// The r-th item of this CTA in the snake order (-1 when there is none).
__device__ __forceinline__ int pair_item_index(int r, int total) {
  const int g = (int)gridDim.x;
  const long long base = (long long)r * g;
  if (base >= total) return -1;
  const long long k = base + ((r & 1) ? g - 1 - (int)blockIdx.x : (int)blockIdx.x);
  return k < total ? (int)k : -2;  // -2: none this round, and none later
}

// kWalk: how an item's KV tiles are enumerated.  kWalkRing: the general
// ring-order walk over num_chunks chunks.  kWalkOne: a single chunk; the
// literal lets the compiler drop the ring-order walk state from every loop,
// which matters at this kernel's register limit (jagged 472 -> 558 TFLOP/s,
// sliding window 943 -> 1040).  kWalkRotated: a ring whose chunks are whole
// tiles, walked as the single chunk rotated to the Q tile's own chunk (the
// ring's tiles, masks and order; long ring 1233 -> 1311).
enum PairWalk : int { kWalkRing = 0, kWalkOne = 1, kWalkRotated = 2 };

template <int D, bool kBf16, int kMode, int kWalk>
// 11 warps put three on three of the four SM sub-partitions (16K registers
// each), so at most 168 registers per thread
__global__ void __launch_bounds__(352, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                        const __grid_constant__ CUtensorMap mv, const PrefillParams p) {
  using C = PairCfg<D>;
  using Walk = std::conditional_t<kWalk == kWalkRotated, LinearWalk, TileWalk>;
  // dense / partial CTAs take one item; the item loops below then run once
  // (a loop the compiler cannot bound costs ~5% in the softmax code)
  constexpr bool kPersistent = kMode == kModeJagged || kMode == kModeWindow;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_q, bar_qe, bar_fin;
  __shared__ uint64_t bar_full[C::NST], bar_empty[C::NST];
  __shared__ uint64_t bar_s[2], bar_p[2], bar_o[2];
  __shared__ uint32_t tmem_slot;
  __shared__ uint32_t abort_flag;
#if ATTN_CHECKED
  // rounds of each stage whose fill its issuer has observed complete
  __shared__ int ring_seen[C::NST];
  if (threadIdx.x < C::NST) ring_seen[threadIdx.x] = 0;
#endif

  const int total = pair_item_count<kMode>(p);
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;  // Q_A, then Q_B
  uint8_t* sKV = smem + 2 * C::Q_BYTES;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_q, 1);
    mbar_init(&bar_qe, 1);
    mbar_init(&bar_fin, 2);  // one commit per MMA issuer
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bar_s[x], 1);
      mbar_init(&bar_p[x], 128);
      mbar_init(&bar_o[x], 1);
    }
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

  // Per item, every role derives the same walk.  Sub-tile x takes part in the
  // tile starting at key `ks` iff it has rows and (causal) its last query
  // sees the tile's first key.
  auto item_walk = [&](const PairItem& it, Walk& walk) -> int {
    const int u_lo = it.st0.q_lo;
    const int u_hi = it.st1.empty() ? it.st0.q_hi : max(it.st0.q_hi, it.st1.q_hi);
    if constexpr (kWalk == kWalkRotated) {
      TileWalk w1;
      w1.init(u_lo, u_hi, it.kv_lo, it.kv_hi, it.q_pos0, it.kv_pos0, p.causal, 1, C::BN,
              kMode == kModeWindow ? p.window : -1);
      walk.init(w1, ring_first_key(u_lo, it.kv_lo, it.kv_hi, it.q_pos0, it.kv_pos0, p.num_chunks), C::BN);
      return walk.n;
    } else {
      walk.init(u_lo, u_hi, it.kv_lo, it.kv_hi, it.q_pos0, it.kv_pos0, p.causal, kWalk == kWalkOne ? 1 : p.num_chunks,
                C::BN, kMode == kModeWindow ? p.window : -1);
      return walk.count();
    }
  };
  auto walk_next = [&](Walk& walk, int& key, int& mask_end) {
    if constexpr (kWalk == kWalkRotated) {
      walk.next(key, mask_end, C::BN);
    } else {
      int ch;
      walk.next(ch, key, mask_end);
    }
  };
  auto active = [&](const PairItem& it, int x, int ks) -> bool {
    const SubTile t = x ? it.st1 : it.st0;
    if (t.empty()) return false;
    if (!p.causal) return true;
    if ((long long)it.kv_pos0 + ks > (long long)it.q_pos0 + t.q_hi - 1) return false;
    // under a sliding window, the tile's last key must reach the first row's window
    return kMode != kModeWindow || (long long)it.kv_pos0 + ks + C::BN - 1 >= (long long)it.q_pos0 + t.q_lo - p.window;
  };

  if (warp == 0) {
    // ========================================================== TMA producer
    if (lane == 0) {
      prefetch_tensormap(&mq);
      prefetch_tensormap(&mk);
      prefetch_tensormap(&mv);
      // a tile load whose coordinates fail the checked build's test loads tile
      // (0, 0, 0, 0) instead, so the pipeline's barriers still complete
      auto load = [&](void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2, int c3, int heads,
                      int rows) {
        if (!check_tile(c0, c1, c2, c3, D, heads, rows, p.B, 256, &g_prefill_status)) c0 = c1 = c2 = c3 = 0;
        tma_load_4d(dst, map, bar, c0, c1, c2, c3);
      };
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;   // K/V slabs issued so far (all items)
      int q_loads = 0;  // items whose Q was loaded
      bool ok = true;
      auto push = [&](const CUtensorMap* map, int hk, int start, int b) -> bool {
        if (!pf_wait(&bar_empty[stage], phase ^ 1u, &abort_flag, 1)) return false;
        uint8_t* dst = sKV + stage * C::SLAB_BYTES;
        mbar_arrive_expect_tx(&bar_full[stage], C::SLAB_BYTES);
        for (int blk = 0; blk < D / 64; ++blk)
          load(dst + blk * C::BLOCK_BYTES, map, &bar_full[stage], blk * 64, hk, start, b, p.h_kv, p.S_kv);
        ++issued;
        if (++stage == C::NST) {
          stage = 0;
          phase ^= 1u;
        }
        return true;
      };
      for (int r = 0; ok && (kPersistent || r == 0); ++r) {
        const int k = pair_item_index(r, total);
        if (k < 0) break;
        const PairUnit un = pair_unit<kMode>(p, k);
        for (int ii = 0; ok && ii < un.n; ++ii) {
          const PairItem it = pair_item<kMode>(p, un.i0 + ii, un.h);
          Walk walk;
          const int n = item_walk(it, walk);
          if (n == 0) continue;
          const int hk = it.st0.h / p.group;
          // Q once the previous item's MMAs are done with the Q buffer, then
          // K/V in the MMA's first-use order: K(0), and per tile V(j), K(j+1)
          Walk kw = walk, vw = walk;
          int s0, me;
          if (q_loads > 0 && !pf_wait(&bar_qe, (uint32_t)((q_loads - 1) & 1), &abort_flag, 4)) {
            ok = false;
            break;
          }
          const int nq = it.st1.empty() ? 1 : 2;
          mbar_arrive_expect_tx(&bar_q, nq * C::Q_BYTES);
          for (int x = 0; x < nq; ++x) {
            const SubTile t = x ? it.st1 : it.st0;
            for (int blk = 0; blk < D / 64; ++blk)
              load(sQ + x * C::Q_BYTES + blk * C::BLOCK_BYTES, &mq, &bar_q, blk * 64, t.h, t.q_lo, it.b, p.h_q, p.S_q);
          }
          ++q_loads;
          walk_next(kw, s0, me);
          ok = push(&mk, hk, s0, it.b);
          if (!ok) break;
          for (int j = 0; ok && j < n; ++j) {
            walk_next(vw, s0, me);
            ok = push(&mv, hk, s0, it.b);
            if (ok && j + 1 < n) {
              walk_next(kw, s0, me);
              ok = push(&mk, hk, s0, it.b);
            }
          }
        }
      }
      if (abort_flag) {
        // copies may still be landing in shared memory: wait for them
        if (q_loads > 0) pf_drain(&bar_q, (uint32_t)((q_loads - 1) & 1));
        const int outstanding = issued < C::NST ? issued : C::NST;
        for (int i = 0; i < outstanding; ++i) {
          const int pos = issued - 1 - i;
          pf_drain(&bar_full[pos % C::NST], (uint32_t)((pos / C::NST) & 1));
        }
      }
    }
  } else if (warp == 1 || warp == 10) {
    // ========================================================== MMA issuers
    // Warp 1 issues the S MMAs, warp 10 the P.V MMAs.  A thread's wait stalls
    // until the tcgen05 work it issued itself has drained from the tensor
    // pipe, so each issuer only waits on the other roles: the S issuer on K
    // stages and, because S_x overwrites the sub-tile's previous P_x in its
    // TMEM buffer and MMAs of different threads are not ordered, on that
    // previous P.V; the P.V issuer on P_x and V stages.
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_f16_f32acc(128, 128, kBf16, false);
      constexpr uint32_t kIdescPV = idesc_f16_f32acc(128, D, kBf16, true);
      const uint32_t sq = smem_u32(sQ);
      const uint32_t skv = smem_u32(sKV);
      const bool s_role = warp == 1;
      int groups[2] = {0, 0};  // S (or P.V) groups issued per sub-tile so far, all items
      int slab0 = 0;           // first K/V slab of the current item
      int q_items = 0;         // items whose Q was consumed
      bool ok = true;
      // slab s (push order K0 V0 K1 V1 ... over all items) lives in stage
      // s % NST, phase (s / NST) & 1.
      // ORDER: the stage's previous fill, slab s - NST, is complete before this
      // wait.  With NST odd it is the other issuer's: for K slab 2m the S issuer
      // has, before this wait, waited for the previous P.V of a sub-tile active
      // on the K tile before, which the P.V issuer issued after waiting for V
      // slab 2(m - (NST + 1) / 2) + 1 = s - NST; for V slab 2m + 1 the P.V
      // issuer has waited for P of the tile before, which its softmax computed
      // from an S MMA issued after the S issuer waited for K slab
      // 2(m - (NST - 1) / 2) = s - NST.  Checked builds verify it (the stage's
      // previous round observed by its issuer) and report a violation as
      // ATTN_ERR_BOUNDS.
      auto wait_slab = [&](int s) -> bool {
#if ATTN_CHECKED
        if (*reinterpret_cast<volatile int*>(&ring_seen[s % C::NST]) < s / C::NST)
          atomicOr(&g_prefill_status, kStatusBounds);
#endif
        if (!pf_wait(&bar_full[s % C::NST], (uint32_t)((s / C::NST) & 1), &abort_flag, 2)) return false;
        tc_fence_after_sync();
#if ATTN_CHECKED
        *reinterpret_cast<volatile int*>(&ring_seen[s % C::NST]) = s / C::NST + 1;
        __threadfence_block();
#endif
        return true;
      };
      for (int r = 0; ok && (kPersistent || r == 0); ++r) {
        const int k = pair_item_index(r, total);
        if (k < 0) break;
        const PairUnit un = pair_unit<kMode>(p, k);
        for (int ii = 0; ok && ii < un.n; ++ii) {
          const PairItem it = pair_item<kMode>(p, un.i0 + ii, un.h);
          Walk walk;
          const int n = item_walk(it, walk);
          if (n == 0) continue;
          if (s_role) {
            if (!pf_wait(&bar_q, (uint32_t)(q_items & 1), &abort_flag, 5)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            ++q_items;
          }
          bool acc[2] = {false, false};  // O_x already holds this item's sum
          for (int j = 0; ok && j < n; ++j) {
            int kstart, me;
            walk_next(walk, kstart, me);
            const bool act[2] = {active(it, 0, kstart), active(it, 1, kstart)};
            const int slab = slab0 + 2 * j + (s_role ? 0 : 1);  // K(j) or V(j)
            ok = wait_slab(slab);
            if (!ok) break;
            const uint32_t stage_addr = skv + (slab % C::NST) * C::SLAB_BYTES;
            // one call per sub-tile, the sub-tile a compile-time constant (as a
            // loop over both with early exits this issue code ran the long ring
            // 4.4 % and the window 2.5 % slower)
            auto serve = [&](auto x_c) {
              constexpr int x = decltype(x_c)::value;
              if (!ok || !act[x]) return;
              const bool last = x == 1 || !act[1];  // last reader of the stage
              if (s_role) {
                if (groups[x] > 0) {
                  // the sub-tile's previous P.V has read its P
                  ok = pf_wait(&bar_o[x], (uint32_t)((groups[x] - 1) & 1), &abort_flag, 11);
                  if (!ok) return;
                  tc_fence_after_sync();
                }
                const uint64_t kdesc = smem_desc_sw128(stage_addr, 16, 1024);
                const uint64_t qdesc = smem_desc_sw128(sq + x * C::Q_BYTES, 16, 1024);
                const uint32_t s_tmem = tmem + static_cast<uint32_t>(x * 128);
                // 16 columns of D per MMA: 32 bytes inside a 128-byte swizzle
                // row, the next 64-column block every four steps
  #pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                  const uint32_t off = (ks / 4) * C::BLOCK_BYTES + (ks % 4) * 32;
                  mma_ss(s_tmem, desc_advance(qdesc, off), desc_advance(kdesc, off), kIdescS, ks != 0);
                }
                if (last) mma_commit(&bar_empty[slab % C::NST]);
                mma_commit(&bar_s[x]);
              } else {
                ok = pf_wait(&bar_p[x], (uint32_t)(groups[x] & 1), &abort_flag, 3);
                if (!ok) return;
                tc_fence_after_sync();
                const uint64_t vdesc = smem_desc_sw128(stage_addr, 16384, 1024);
                const uint32_t p_tmem = tmem + static_cast<uint32_t>(x * 128);
                const uint32_t o_tmem = tmem + C::O_COL + static_cast<uint32_t>(x * D);
                // 16 keys of V (16 rows of 256 bytes, two swizzle atoms) per MMA
  #pragma unroll
                for (int ks = 0; ks < C::BN / 16; ++ks)
                  mma_ts(o_tmem, p_tmem + ks * 8, desc_advance(vdesc, ks * 2048), kIdescPV,
                         (ks > 0 || acc[x]) ? 1u : 0u);
                acc[x] = true;
                if (last) mma_commit(&bar_empty[slab % C::NST]);
                mma_commit(&bar_o[x]);
              }
              ++groups[x];
            };
            serve(std::integral_constant<int, 0>{});
            serve(std::integral_constant<int, 1>{});
          }
          if (!ok) break;
          // the item's S MMAs, the last readers of its Q, release the Q buffer
          if (s_role) mma_commit(&bar_qe);
          slab0 += 2 * n;
        }
      }
      // every MMA either issuer issued must finish before TMEM is released
      mma_commit(&bar_fin);
      pf_drain(&bar_fin, 0);
    }
  } else {
    // ========================================================== softmax + epilogue
    const int x = (warp - 2) >> 2;  // sub-tile of this warpgroup
    const int wq = warp & 3;        // TMEM lane quarter this warp may access
    const int row = wq * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t scol = lane_addr + static_cast<uint32_t>(x * 128);
    const uint32_t ocol = lane_addr + C::O_COL + static_cast<uint32_t>(x * D);
    const float c = p.scale_log2;  // > 0
    const uint64_t c2 = f2_make(c, c);
    const uint32_t ninf = __float_as_uint(-CUDART_INF_F);
    int cnt = 0;  // tiles this sub-tile took part in (all items) = its P.V groups
    bool ok = true;
    for (int r = 0; ok && (kPersistent || r == 0); ++r) {
      const int k = pair_item_index(r, total);
      if (k < 0) break;
      const PairUnit un = pair_unit<kMode>(p, k);
      for (int ii = 0; ok && ii < un.n; ++ii) {
        const PairItem it = pair_item<kMode>(p, un.i0 + ii, un.h);
        Walk walk;
        const int n = item_walk(it, walk);
        const SubTile me_t = x ? it.st1 : it.st0;
        const int q_row = me_t.q_lo + row;
        float m_run = -CUDART_INF_F;  // reference max (exp2 domain), raised lazily
        float l_run = 0.f;            // sum of exp2(x - m_run) in fp32: the triplet's l and the LSE
        float lr_run = 0.f;           // sum of the rounded P the MMA multiplies V by: normalises O
        float m_max = -CUDART_INF_F;  // true running max (partial mode)
        int cnt_item = 0;             // tiles of this item this sub-tile took part in
        for (int j = 0; j < n; ++j) {
          int kstart, mend;
          walk_next(walk, kstart, mend);
          if (!active(it, x, kstart)) continue;
          if (!pf_wait(&bar_s[x], (uint32_t)(cnt & 1), &abort_flag, 6)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          // S_x(j) was issued after this sub-tile's previous P.V by the same
          // thread, so its completion also means that P.V has finished: O may
          // be rescaled without waiting on bar_o.
          constexpr bool win = kMode == kModeWindow;
          const bool need_mask =
              (kstart + C::BN > mend) ||
              (p.causal && ((long long)it.kv_pos0 + kstart + C::BN - 1 > (long long)it.q_pos0 + me_t.q_lo)) ||
              (win && (long long)it.kv_pos0 + kstart < (long long)it.q_pos0 + me_t.q_hi - 1 - p.window);
          long long lim = C::BN;  // key kstart + i is visible iff flo <= i < lim
          long long flo = 0;
          int ilim = C::BN, iflo = 0;  // the same limits clamped to the tile
          if (need_mask) {
            lim = (long long)mend - kstart;
            if (p.causal) {
              const long long lc = (long long)it.q_pos0 + q_row - it.kv_pos0 - kstart + 1;
              lim = lc < lim ? lc : lim;
              if (win) flo = lc - 1 - p.window;
            }
            ilim = clamp_limit(lim, C::BN);
            iflo = clamp_limit(flo, C::BN);
          }
          // the first 64 columns are reduced while the second pair of loads is in flight
          uint32_t r0[32], r1[32], r2[32], r3[32];
          tmem_ld32(scol, r0);
          tmem_ld32(scol + 32, r1);
          tmem_ld_wait(r0);
          tmem_ld_wait(r1);
          tmem_ld32(scol + 64, r2);
          tmem_ld32(scol + 96, r3);
          // the persistent modes (many masked tiles) take 32-bit chunk masks;
          // the other walks keep per-score compares, which allocate better there
          if (need_mask) {
            if constexpr (kPersistent) {
              apply_mask(r0, chunk_mask(0, iflo, ilim), ninf);
              apply_mask(r1, chunk_mask(32, iflo, ilim), ninf);
            } else {
  #pragma unroll
              for (int i = 0; i < 32; ++i) {
                if (i >= lim || i < flo) r0[i] = ninf;
                if (i + 32 >= lim || i + 32 < flo) r1[i] = ninf;
              }
            }
          }
          float mx8[8];
  #pragma unroll
          for (int i = 0; i < 8; ++i) {
            mx8[i] = fmax3(__uint_as_float(r0[i]), __uint_as_float(r0[i + 8]), __uint_as_float(r0[i + 16]));
            mx8[i] = fmax3(mx8[i], __uint_as_float(r0[i + 24]), __uint_as_float(r1[i]));
            mx8[i] = fmax3(mx8[i], __uint_as_float(r1[i + 8]), __uint_as_float(r1[i + 16]));
          }
          tmem_ld_wait(r2);
          tmem_ld_wait(r3);
          if (need_mask) {
            if constexpr (kPersistent) {
              apply_mask(r2, chunk_mask(64, iflo, ilim), ninf);
              apply_mask(r3, chunk_mask(96, iflo, ilim), ninf);
            } else {
  #pragma unroll
              for (int i = 0; i < 32; ++i) {
                if (i + 64 >= lim || i + 64 < flo) r2[i] = ninf;
                if (i + 96 >= lim || i + 96 < flo) r3[i] = ninf;
              }
            }
          }
  #pragma unroll
          for (int i = 0; i < 8; ++i) {
            mx8[i] = fmax3(mx8[i], __uint_as_float(r1[i + 24]), __uint_as_float(r2[i]));
            mx8[i] = fmax3(mx8[i], __uint_as_float(r2[i + 8]), __uint_as_float(r2[i + 16]));
            mx8[i] = fmax3(mx8[i], __uint_as_float(r2[i + 24]), __uint_as_float(r3[i]));
            mx8[i] = fmax3(mx8[i], __uint_as_float(r3[i + 8]), __uint_as_float(r3[i + 16]));
            mx8[i] = fmaxf(mx8[i], __uint_as_float(r3[i + 24]));
          }
          const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
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
          const float neg_m = m_run == -CUDART_INF_F ? 0.f : -m_run;
          const uint64_t nm2 = f2_make(neg_m, neg_m);
          uint64_t sum2 = f2_make(0.f, 0.f);
          float sr[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // rounded weights, 8 chains
          uint32_t pk[16];
          auto pack_chunk = [&](uint32_t (&rr)[32], uint32_t col) {
  #pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 e = f2_split(f2_fma(f2_make_u(rr[2 * i], rr[2 * i + 1]), c2, nm2));
              const float p0 = fast_exp2(e.x), p1 = fast_exp2(e.y);
              pk[i] = pack_half2<kBf16>(p0, p1);
              sum2 = f2_add(sum2, f2_make(p0, p1));
              // O is normalised by the sum of the rounded weights it was built
              // from, so O / l is a weighted mean with consistent weights
              add_half2_to_f32<kBf16>(sr[2 * (i & 3)], sr[2 * (i & 3) + 1], pk[i]);
            }
            tmem_st16(scol + col, pk);
          };
          // P overwrites the first 64 columns of S, already in registers
          pack_chunk(r0, 0);
          pack_chunk(r1, 16);
          // O (complete up to the previous tile, see above) is rescaled before
          // P(j) is published
          if (cnt_item > 0 && __any_sync(0xffffffffu, raise)) {
  #pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t o[32];
              tmem_ld32(ocol + cc * 32, o);
              tmem_ld_wait(o);
  #pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(ocol + cc * 32, o);
            }
          }
          pack_chunk(r2, 32);
          pack_chunk(r3, 48);
          const float2 sv = f2_split(sum2);
          l_run += sv.x + sv.y;
          lr_run += ((sr[0] + sr[1]) + (sr[2] + sr[3])) + ((sr[4] + sr[5]) + (sr[6] + sr[7]));
          tmem_st_wait();
          tc_fence_before_sync();
          mbar_arrive(&bar_p[x]);
          ++cnt;
          ++cnt_item;
        }
        if (!ok) break;
        if (cnt_item > 0) {
          // the item's last P.V of this sub-tile (earlier ones are done, see above)
          if (!pf_wait(&bar_o[x], (uint32_t)((cnt - 1) & 1), &abort_flag, 8)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
        }
        const size_t row_idx = ((size_t)it.b * p.S_q + q_row) * p.h_q + me_t.h;
        const size_t lse_idx = ((size_t)it.b * p.h_q + me_t.h) * p.S_q + q_row;
        const long long rows_all = (long long)p.B * p.S_q * p.h_q;
        const bool row_valid = q_row < me_t.q_hi && check_index((long long)row_idx, rows_all, &g_prefill_status) &&
                               check_index((long long)lse_idx, rows_all, &g_prefill_status);
        if constexpr (kPersistent) {
          // persistent launches (short items, so the epilogue weighs): O read
          // with two TMEM loads in flight (jagged +1.4 %, the sliding window
          // +0.4 %); dense launches keep one load at a time (the long ring ran
          // 1 % slower with the pipelined form)
          constexpr float kLn2 = 0.693147180559945309f;
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
          const bool o_v8 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
          auto emit = [&](int cc, const uint32_t(&o)[32]) {
            if (!row_valid) return;
            if constexpr (kMode != kModePartial) {
              uint32_t w[16];
    #pragma unroll
              for (int i = 0; i < 16; ++i)
                w[i] = pack_half2<kBf16>(__uint_as_float(o[2 * i]) * so, __uint_as_float(o[2 * i + 1]) * so);
              uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + row_idx * D + cc * 32;
              // a warp's store touches 32 rows: 32-byte pieces halve the
              // requests of 16-byte ones (the output's base decides)
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
          if (cnt_item > 0) {
            // two chunks of 32 columns in flight, chunk c + 1 loading while chunk
            // c is normalised and stored
            uint32_t oa[32], ob[32];
            tmem_ld32(ocol, oa);
            tmem_ld_wait(oa);
    #pragma unroll 1
            for (int cc = 0; cc < D / 32; cc += 2) {
              tmem_ld32(ocol + (cc + 1) * 32, ob);
              emit(cc, oa);
              tmem_ld_wait(ob);
              if (cc + 2 < D / 32) tmem_ld32(ocol + (cc + 2) * 32, oa);
              emit(cc + 1, ob);
              if (cc + 2 < D / 32) tmem_ld_wait(oa);
            }
          } else {
            // no visible key: O = 0 (and LSE = -inf)
            uint32_t z[32];
    #pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0u;
    #pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) emit(cc, z);
          }
          if constexpr (kMode != kModePartial) {
            if (p.lse != nullptr && row_valid)
              p.lse[lse_idx] = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -CUDART_INF_F;
          } else if (row_valid) {
            p.m_out[lse_idx] = any ? m_max * kLn2 : -CUDART_INF_F;
            p.l_out[lse_idx] = any ? l_run * f : 0.f;
          }
        } else {
          constexpr float kLn2 = 0.693147180559945309f;
          if constexpr (kMode != kModePartial) {
            const float inv_l = lr_run > 0.f ? 1.f / lr_run : 0.f;
            uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + row_idx * D;
            const bool o_v8 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
    #pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t o[32];
              if (cnt_item > 0) {
                tmem_ld32(ocol + cc * 32, o);
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
                // a warp's store touches 32 rows: 32-byte pieces halve the
                // requests of 16-byte ones (the output's base decides)
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
            if (p.lse != nullptr && row_valid)
              p.lse[lse_idx] = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -CUDART_INF_F;
          } else {
            const bool any = l_run > 0.f && m_max != -CUDART_INF_F;
            const float f = any ? fast_exp2(m_run - m_max) : 0.f;  // re-reference to the true max
            // O re-weighted so that O / l equals the consistently normalised O_acc / lr
            const float fo = any ? f * (l_run / lr_run) : 0.f;
            float* orow = p.o_part + row_idx * D;
    #pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t o[32];
              if (cnt_item > 0) {
                tmem_ld32(ocol + cc * 32, o);
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
            if (row_valid) {
              p.m_out[lse_idx] = any ? m_max * kLn2 : -CUDART_INF_F;
              p.l_out[lse_idx] = any ? l_run * f : 0.f;
            }
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool kBf16, int kMode, int kWalk>
attn_status_t launch_pair_variant(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                  const CUtensorMap& mv, dim3 grid, cudaStream_t s) {
  using C = PairCfg<D>;
  auto kern = prefill_pair_kernel<D, kBf16, kMode, kWalk>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
    return ATTN_ERR_CUDA;
  kern<<<grid, C::THREADS, C::SMEM_BYTES, s>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Dense and window launches with one chunk take the single-chunk
// instantiations, with ring chunks of whole tiles the rotated ones, otherwise
// the general ring walk; every partial and jagged launch (always one KV range)
// takes the single-chunk instantiation.
template <int D, bool kBf16>
attn_status_t launch_pair_typed(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                const CUtensorMap& mv, int mode, dim3 grid, cudaStream_t s) {
  const bool one = p.num_chunks == 1;
  const bool rotated = ring_walk_is_rotation(p.kv_lo, p.kv_hi, p.num_chunks, PairCfg<D>::BN);
  switch (mode) {
    case kModeDense:
      return one       ? launch_pair_variant<D, kBf16, kModeDense, kWalkOne>(p, mq, mk, mv, grid, s)
             : rotated ? launch_pair_variant<D, kBf16, kModeDense, kWalkRotated>(p, mq, mk, mv, grid, s)
                       : launch_pair_variant<D, kBf16, kModeDense, kWalkRing>(p, mq, mk, mv, grid, s);
    case kModeWindow:
      return one       ? launch_pair_variant<D, kBf16, kModeWindow, kWalkOne>(p, mq, mk, mv, grid, s)
             : rotated ? launch_pair_variant<D, kBf16, kModeWindow, kWalkRotated>(p, mq, mk, mv, grid, s)
                       : launch_pair_variant<D, kBf16, kModeWindow, kWalkRing>(p, mq, mk, mv, grid, s);
    case kModePartial:
      return one ? launch_pair_variant<D, kBf16, kModePartial, kWalkOne>(p, mq, mk, mv, grid, s) : ATTN_ERR_INVALID_ARG;
    case kModeJagged:
      return one ? launch_pair_variant<D, kBf16, kModeJagged, kWalkOne>(p, mq, mk, mv, grid, s) : ATTN_ERR_INVALID_ARG;
  }
  return ATTN_ERR_INVALID_ARG;
}

template <int D>
attn_status_t launch_pair_dispatch(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                   const CUtensorMap& mv, int mode, bool bf16, dim3 grid, cudaStream_t s) {
  return bf16 ? launch_pair_typed<D, true>(p, mq, mk, mv, mode, grid, s)
              : launch_pair_typed<D, false>(p, mq, mk, mv, mode, grid, s);
}

}  // namespace attn
