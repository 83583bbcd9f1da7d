// Tile schedule shared by host and device: which KV tiles one Q tile visits.
//
// "[pallas] Support dependent Tile.end bounds in Pallas" (opening example,
// "Unroll lowering"): the inner KV loop of a Q tile runs over
// [kv_begin, min(kv_end, tile_q.end)) in tiles of block_k keys, i.e.
// trip_count = cdiv(active_end - begin, block_k) tiles, the last one masked by
// indices_k < active_end.  Fully masked tiles are never visited (pruned).
//
// Sliding window (causal, window >= 0): a key is visible to a query iff
// q - window <= k <= q, the dependent lower bound max(kv_begin, tile_q.begin -
// window) that the same page ("Scalar minimum") defers to sliding-window
// support.  A chunk's tiles still start on its block_n grid; the walk starts at
// the tile holding the first key the Q tile's first row can see.
//
// "kernbench2 _gqa_prefill_long.py" (module docstring, P6b; ring loop): a
// unit that starts on its own KV block and receives from its east neighbour
// sees blocks (c + t) mod C.  Here the C chunks of one KV range are walked in
// that order inside one kernel, starting at the chunk that holds the Q tile's
// first position; a chunk whose visible part is empty is skipped (the causal
// step-skip the page lists as missing).
#pragma once

#include <limits.h>

namespace attn {

struct TileWalk {
  // query rows [q_lo, q_hi) at positions q_pos0 + row; keys [kv_lo, kv_hi) at
  // positions kv_pos0 + key (each in its own tensor's index space)
  int kv_lo, kv_hi, block_n, num_chunks;
  int chunk_len, c0;
  int key_limit;  // keys with index >= key_limit are invisible to every row of the tile
  int key_floor;  // keys with index < key_floor are invisible to every row (sliding window)
  // cursor
  int t, chunk, cur, end;

  __host__ __device__ void init(int q_lo, int q_hi, int kv_lo_, int kv_hi_, int q_pos0, int kv_pos0, int causal,
                                int num_chunks_, int block_n_, int window = -1) {
    kv_lo = kv_lo_;
    kv_hi = kv_hi_;
    block_n = block_n_;
    num_chunks = num_chunks_ < 1 ? 1 : num_chunks_;
    const int len = kv_hi - kv_lo;
    chunk_len = len > 0 ? (len + num_chunks - 1) / num_chunks : 1;
    const long long rel = (long long)q_pos0 + q_lo - ((long long)kv_pos0 + kv_lo);
    long long c = rel <= 0 ? 0 : rel / chunk_len;
    c0 = (int)(c > num_chunks - 1 ? num_chunks - 1 : c);
    if (causal) {
      // the tile's last query sits at q_pos0 + q_hi - 1; key index k is visible
      // to it iff kv_pos0 + k <= q_pos0 + q_hi - 1
      long long lim = (long long)q_pos0 + q_hi - kv_pos0;
      key_limit = q_hi <= q_lo ? INT_MIN : (int)(lim > INT_MAX ? INT_MAX : (lim < INT_MIN ? INT_MIN : lim));
    } else {
      key_limit = q_hi <= q_lo ? INT_MIN : INT_MAX;
    }
    key_floor = INT_MIN;
    if (causal && window >= 0) {
      // the tile's first query sits at q_pos0 + q_lo and sees keys from position
      // q_pos0 + q_lo - window on
      const long long fl = (long long)q_pos0 + q_lo - window - kv_pos0;
      key_floor = (int)(fl > INT_MAX ? INT_MAX : (fl < INT_MIN ? INT_MIN : fl));
    }
    t = 0;
    open_chunk();
  }

  // Moves to the next chunk (from t on) with a non-empty visible part.
  __host__ __device__ void open_chunk() {
    while (t < num_chunks) {
      chunk = (c0 + t) % num_chunks;
      const long long lo_ll = (long long)kv_lo + (long long)chunk * chunk_len;
      const int lo = (int)(lo_ll < kv_hi ? lo_ll : kv_hi);
      const long long hi_ll = lo_ll + chunk_len;
      const int hi = (int)(hi_ll < kv_hi ? hi_ll : kv_hi);
      end = hi < key_limit ? hi : key_limit;  // min(chunk_end, tile_q.end)
      int start = lo;
      if (key_floor > lo) {  // first tile of the chunk's grid that holds a key >= key_floor
        const long long skip = ((long long)key_floor - lo) / block_n;
        const long long st = lo + skip * block_n;
        start = (int)(st < end ? st : end);
      }
      if (end > start && key_floor < end) {
        cur = start;
        return;
      }
      ++t;
    }
  }

  // Next visited tile: keys [start, start + block_n) of chunk `c`; keys at or
  // beyond mask_end are excluded by the tail mask.
  __host__ __device__ bool next(int& c, int& start, int& mask_end) {
    if (t >= num_chunks) return false;
    c = chunk;
    start = cur;
    mask_end = end;
    cur += block_n;
    if (cur >= end) {
      ++t;
      open_chunk();
    }
    return true;
  }

  // Total number of tiles the walk visits (closed form per chunk).
  __host__ __device__ int count() const {
    TileWalk w = *this;
    int n = 0;
    while (w.t < w.num_chunks) {
      n += (w.end - w.cur + w.block_n - 1) / w.block_n;
      ++w.t;
      w.open_chunk();
    }
    return n;
  }
};

// Whether the ring walk of num_chunks chunks over [kv_lo, kv_hi) is a rotation
// of the single-chunk walk: it is when the chunk length is a multiple of
// block_n.  Every chunk then starts on the range's block_n grid, so the ring
// visits the single-chunk walk's tiles, with the same tail masks (no tile spans
// two chunks), in the order: from the first tile of chunk c0 (the chunk of the
// Q tile's first position) up, then from the first visible tile up to chunk c0.
// Chunks past the causal limit hold no visible tile, and the chunks after c0
// and the ones before it are each taken in ascending order, as in the ring.
__host__ __device__ inline bool ring_walk_is_rotation(int kv_lo, int kv_hi, int num_chunks, int block_n) {
  if (num_chunks <= 1) return false;
  const int len = kv_hi - kv_lo;
  const int chunk_len = len > 0 ? (len + num_chunks - 1) / num_chunks : 1;
  return chunk_len % block_n == 0;
}

// First key of chunk c0 (the chunk that holds the Q tile's first position), as
// TileWalk::init chooses it.
__host__ __device__ inline int ring_first_key(int q_lo, int kv_lo, int kv_hi, int q_pos0, int kv_pos0,
                                              int num_chunks) {
  const int len = kv_hi - kv_lo;
  const int chunk_len = len > 0 ? (len + num_chunks - 1) / num_chunks : 1;
  const long long rel = (long long)q_pos0 + q_lo - ((long long)kv_pos0 + kv_lo);
  long long c = rel <= 0 ? 0 : rel / chunk_len;
  if (c > num_chunks - 1) c = num_chunks - 1;
  const long long k = (long long)kv_lo + c * chunk_len;
  return (int)(k < kv_hi ? k : kv_hi);
}

// The single-chunk walk's tiles [start, end), taken from the tile at key
// `first` up and then from `start` up to it: with first = start it is the
// single-chunk walk itself, with first = ring_first_key() the ring walk when
// ring_walk_is_rotation() holds.  Three integers of state, for kernels whose
// registers are scarce.
struct LinearWalk {
  int cur, start, end;
  int n;  // tiles

  __host__ __device__ void init(const TileWalk& one_chunk, int first, int block_n) {
    if (one_chunk.t >= one_chunk.num_chunks) {  // nothing visible
      start = end = cur = 0;
      n = 0;
      return;
    }
    start = one_chunk.cur;
    end = one_chunk.end;
    n = (end - start + block_n - 1) / block_n;
    // first is on the start's block_n grid when it lies inside the range
    cur = first > start && first < end ? first : start;
  }

  // Next tile: keys [key, key + block_n), the tail mask at mask_end.  Call it
  // n times.
  __host__ __device__ void next(int& key, int& mask_end, int block_n) {
    key = cur;
    mask_end = end;
    cur += block_n;
    if (cur >= end) cur = start;
  }
};

// Work units of a head-dim-256 dense / partial / window launch, which runs on
// CTA pairs: a pair item is 256 query rows (two consecutive 128-row Q tiles of
// one head, or with pair_heads one Q tile of two query heads), and a unit is
// up to two items of one (batch, head or head pair).
__host__ __device__ inline long long cta2_units(int B, int S_q, int h_q, int pair_heads) {
  const int n_qt = (S_q + 127) / 128;
  const int n_it = pair_heads ? n_qt : (n_qt + 1) / 2;
  const int n_y = pair_heads ? h_q / 2 : h_q;
  return (long long)((n_it + 1) / 2) * n_y * B;
}

}  // namespace attn
