"""Integer oracle for the tile schedule: which KV tiles a Q tile visits.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources (page title, section):
  * "[pallas] Support dependent Tile.end bounds in Pallas", opening example:
    the inner KV loop runs over hl.tile(kv_begin, min(kv_end, tile_q.end)).
  * same page, "Unroll lowering": trip_count = cdiv(active_end - begin, block_k)
    and the tail mask indices_k < active_end.
  * same page, "Flattened worklists": ordered_begin = range_start[wid],
    source_end = ordered_begin + range_len[wid],
    compact_end = tile_start[wid] + tile_extent[wid],
    compute_end = min(source_end, compact_end) drives the trip count.
  * same page, review thread: the jagged KV end is seq_offsets[seq_idx + 1].
  * "kernbench2 _gqa_prefill_long.py", module docstring (P6b) and the ring
    loop: over C-1 steps a unit that starts on its own KV block receives the
    block of its east neighbour, so it sees blocks (c + t) mod C; its
    "Deviations" list names causal step-skip as the missing piece.

The functions here decide tile visits by BRUTE FORCE over (query, key) pairs:
a tile is visited iff it holds at least one visible pair.  The closed-form
trip counts of the pages are what the library implements; tests check that
the two agree exactly.
"""

from __future__ import annotations

import numpy as np


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


def pair_visible_in(q_lo: int, q_hi: int, k_lo: int, k_hi: int, causal: bool,
                    q_pos0: int = 0, kv_pos0: int = 0, window: int | None = None) -> bool:
    """True iff some query in [q_lo, q_hi) sees some key in [k_lo, k_hi).

    With a sliding window (causal only) key position p is visible to query
    position i iff i - window <= p <= i.
    """
    if q_hi <= q_lo or k_hi <= k_lo:
        return False
    if not causal:
        return True
    qpos = np.arange(q_lo, q_hi, dtype=np.int64) + q_pos0
    kpos = np.arange(k_lo, k_hi, dtype=np.int64) + kv_pos0
    vis = kpos[None, :] <= qpos[:, None]
    if window is not None:
        vis &= kpos[None, :] >= qpos[:, None] - window
    return bool(vis.any())


def ring_chunks(kv_lo: int, kv_hi: int, num_chunks: int):
    """[kv_lo, kv_hi) cut into num_chunks ranges of ceil(len / C) keys (last ones may be empty)."""
    step = max(1, cdiv(kv_hi - kv_lo, num_chunks))
    return [(min(kv_lo + c * step, kv_hi), min(kv_lo + (c + 1) * step, kv_hi))
            for c in range(num_chunks)], step


def ring_start_chunk(q_lo: int, kv_lo: int, kv_hi: int, num_chunks: int,
                     q_pos0: int = 0, kv_pos0: int = 0) -> int:
    """The chunk holding the Q tile's first position (its "own" block), clamped to [0, C)."""
    _, step = ring_chunks(kv_lo, kv_hi, num_chunks)
    rel = (q_pos0 + q_lo) - (kv_pos0 + kv_lo)
    return int(min(max(rel // step, 0), num_chunks - 1))


def tile_walk(q_lo: int, q_hi: int, kv_lo: int, kv_hi: int, block_n: int, causal: bool,
              num_chunks: int = 1, q_pos0: int = 0, kv_pos0: int = 0, window: int | None = None):
    """Ordered KV tiles visited by the Q tile [q_lo, q_hi).

    Chunks are walked in ring order starting at the Q tile's own chunk; inside
    a chunk, tiles of block_n keys start at the chunk start.  A tile is kept iff
    it holds a visible pair (brute force); a chunk with no kept tile is skipped.
    Returns a list of (chunk, tile_start, tile_stop), tile_stop clipped to the
    chunk end.
    """
    chunks, _ = ring_chunks(kv_lo, kv_hi, num_chunks)
    c0 = ring_start_chunk(q_lo, kv_lo, kv_hi, num_chunks, q_pos0, kv_pos0)
    walk = []
    for t in range(num_chunks):
        c = (c0 + t) % num_chunks
        lo, hi = chunks[c]
        start = lo
        while start < hi:
            stop = min(start + block_n, hi)
            if pair_visible_in(q_lo, q_hi, start, stop, causal, q_pos0, kv_pos0, window):
                walk.append((c, start, stop))
            start += block_n
    return walk


def dense_work_items(S_q: int, block_m: int):
    """Q tiles [t*BM, min((t+1)*BM, S_q)) of one (batch, head)."""
    return [(t * block_m, min((t + 1) * block_m, S_q)) for t in range(cdiv(S_q, block_m))]


def jagged_worklist(seq_offsets, block_m: int, block_n: int, causal: bool = True):
    """Flattened jagged worklist: one item per (sequence, Q tile).

    Fields follow the pages' flattened-worklist names.  The trip count is
    counted by brute force (tiles of the source range holding a visible
    pair); the tests check it equals cdiv(compute_end - ordered_begin, block_n).
    Returns items sorted by (seq, tile).
    """
    offs = np.asarray(seq_offsets, dtype=np.int64)
    items = []
    for b in range(offs.size - 1):
        begin, end = int(offs[b]), int(offs[b + 1])
        length = end - begin
        for t in range(cdiv(length, block_m)):
            tile_start = begin + t * block_m
            tile_extent = min(block_m, end - tile_start)
            source_end = begin + length
            compact_end = tile_start + tile_extent
            compute_end = min(source_end, compact_end) if causal else source_end
            walk = tile_walk(tile_start, compact_end, begin, end, block_n, causal)
            trip = len(walk)
            items.append(dict(seq=b, tile=t, ordered_begin=begin, range_len=length,
                              tile_start=tile_start, tile_extent=tile_extent,
                              compute_end=compute_end, trip=trip))
    return items


def visited_tile_count_dense_causal(S: int, block: int) -> int:
    """Closed form: T(T+1)/2 tiles of one (batch, head) for S = T * block, BM = BN."""
    t = cdiv(S, block)
    return t * (t + 1) // 2
