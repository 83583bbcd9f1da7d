"""Pins of the integer schedule oracle (CPU only).

The oracle decides tile visits by brute force over (query, key) pairs.  Here it
is pinned to hand-derived walks (tests/golden), to closed-form tile counts and to
the pages' closed-form trip count cdiv(min(kv_end, tile_q.end) - begin, block_k).
"""

import numpy as np
import pytest

from oracle import schedule as S


def test_golden_schedule(golden):
    for case in golden["schedule"]:
        if "walks" in case:
            items = S.dense_work_items(case["S"], case["block_m"])
            walks = [S.tile_walk(lo, hi, 0, case["S"], case["block_n"], case["causal"],
                                 case["num_chunks"]) for lo, hi in items]
            assert [[list(t) for t in w] for w in walks] == case["walks"], case["name"]
        else:
            lo, hi = case["q_tile"]
            w = S.tile_walk(lo, hi, 0, case["S"], case["block_n"], case["causal"], case["num_chunks"])
            assert [list(t) for t in w] == case["walk"], case["name"]


def test_dense_causal_tile_count_closed_form():
    # 4096 keys in 128-tiles: 32*33/2 = 528 of 1024 tiles per (batch, head)
    total = sum(len(S.tile_walk(lo, hi, 0, 4096, 128, True)) for lo, hi in S.dense_work_items(4096, 128))
    assert total == 528 == S.visited_tile_count_dense_causal(4096, 128)


def test_ring_walk_counts_closed_form():
    """S=32768, C=8 chunks: 256 Q tiles visit 256*257/2 = 32896 tiles and on average 4.5 chunks."""
    Sq, C, blk = 32768, 8, 128
    tiles = 0
    chunk_steps = 0
    for lo, hi in S.dense_work_items(Sq, blk):
        # count per chunk without materialising every pair: a tile is visited
        # iff its first key is <= the tile's last query (checked by brute force below)
        w = S.tile_walk(lo, hi, 0, Sq, blk, True, C) if lo % (16 * blk) == 0 else None
        c0 = lo // (Sq // C)
        n_tiles = hi // blk
        if w is not None:
            assert len(w) == n_tiles
            assert [c for c, _, _ in w][0] == c0
            assert len({c for c, _, _ in w}) == c0 + 1
        tiles += n_tiles
        chunk_steps += c0 + 1
    assert tiles == 32896
    assert chunk_steps / 256 == 4.5


@pytest.mark.parametrize("seed", range(40))
def test_trip_count_formula_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    S_q = int(rng.integers(1, 700))
    S_kv = S_q if rng.random() < 0.6 else int(rng.integers(1, 700))
    bm = int(rng.choice([64, 128]))
    bn = int(rng.choice([64, 128]))
    causal = bool(rng.random() < 0.7)
    C = int(rng.integers(1, 6))
    chunks, step = S.ring_chunks(0, S_kv, C)
    for lo, hi in S.dense_work_items(S_q, bm):
        w = S.tile_walk(lo, hi, 0, S_kv, bn, causal, C)
        c0 = S.ring_start_chunk(lo, 0, S_kv, C)
        expect = []
        for t in range(C):
            c = (c0 + t) % C
            c_lo, c_hi = chunks[c]
            end = min(c_hi, hi) if causal else c_hi  # min(kv_end, tile_q.end)
            trip = S.cdiv(end - c_lo, bn) if end > c_lo else 0
            expect += [(c, c_lo + i * bn, min(c_lo + (i + 1) * bn, c_hi)) for i in range(trip)]
        assert w == expect


def test_jagged_worklist_fields_and_trip_counts():
    offs = np.array([0, 5, 5, 300, 301, 700])
    items = S.jagged_worklist(offs, 128, 128, causal=True)
    # lengths 5, 0, 295, 1, 399 -> 1 + 0 + 3 + 1 + 4 Q tiles
    assert len(items) == 9
    assert sum(it["seq"] == 1 for it in items) == 0
    for it in items:
        assert it["trip"] == S.cdiv(it["compute_end"] - it["ordered_begin"], 128)
        assert it["trip"] == it["tile"] + 1  # BM = BN, causal
        assert it["compute_end"] == min(it["ordered_begin"] + it["range_len"],
                                        it["tile_start"] + it["tile_extent"])
    last = [it for it in items if it["seq"] == 4][-1]
    assert (last["tile_start"], last["tile_extent"], last["compute_end"]) == (301 + 384, 15, 700)
    nc = S.jagged_worklist(offs, 128, 128, causal=False)
    assert all(it["trip"] == S.cdiv(it["range_len"], 128) for it in nc)


def test_jagged_tile_count_closed_form():
    rng = np.random.default_rng(0)
    lens = rng.integers(64, 1025, 50)
    offs = np.concatenate([[0], np.cumsum(lens)])
    items = S.jagged_worklist(offs, 128, 128)
    n = (lens + 127) // 128
    assert len(items) == int(n.sum())
    assert sum(it["trip"] for it in items) == int((n * (n + 1) // 2).sum())
