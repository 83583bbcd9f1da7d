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

}  // namespace attn
