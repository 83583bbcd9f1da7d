"""C-ABI checks that need no GPU: the library loads, exports every declared
symbol, rejects bad arguments on the host, and its tile scheduler (the same code
the kernels run) matches the oracle's brute-force walk bit for bit."""

import ctypes
import os
import re

import numpy as np
import pytest

import ring_attention_online_gb300 as ra
from oracle import schedule as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(ra.library_path()):
        from ring_attention_online_gb300 import build
        build.build()
    return ra.load_library()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_symbols()
    assert len(names) >= 10
    for name in names:
        assert hasattr(lib, name), name


def test_binding_names_match_the_abi():
    for name in _declared_symbols():
        assert callable(getattr(ra, name)), name


FAKE = ctypes.c_void_p(0x10000)  # aligned, never dereferenced: validation fails first


def test_prefill_validation(lib):
    ok_args = [FAKE, FAKE, FAKE, FAKE, None, 1, 128, 128, 2, 1, 128, 1, 0.1, 1, 1, None]

    def call(**over):
        a = list(ok_args)
        for i, v in over.items():
            a[int(i[1:])] = v
        return lib.attn_prefill(*a)

    assert call(a0=None) == 1                    # null q
    assert call(a3=None) == 1                    # null o
    assert call(a8=2, a9=3) == 1                 # h_q % h_kv != 0
    assert call(a10=96) == 2                     # D outside {64,128,256}
    assert call(a11=7) == 1                      # bad dtype
    assert call(a12=0.0) == 1                    # scale must be > 0
    assert call(a12=float("nan")) == 1
    assert call(a13=2) == 1                      # causal must be 0/1
    assert call(a14=0) == 1                      # num_chunks >= 1
    assert call(a0=ctypes.c_void_p(0x10008)) == 1  # misaligned
    assert call(a5=-1) == 1
    assert call(a5=0) == 0                       # empty batch: no-op
    assert call(a6=0) == 0                       # empty query: no-op


def test_partial_merge_jagged_decode_validation(lib):
    assert lib.attn_partial(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 8, 1, 1, 64, 0, 0.5, 0, 0, 5, 3, None) == 1
    assert lib.attn_partial(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 8, 1, 1, 64, 0, 0.5, 0, 0, 0, 9, None) == 1
    assert lib.attn_partial(FAKE, FAKE, FAKE, None, FAKE, FAKE, 1, 4, 8, 1, 1, 64, 0, 0.5, 0, 0, 0, 8, None) == 1
    assert lib.attn_merge(FAKE, FAKE, FAKE, 0, 1, 1, 1, 64, FAKE, 0, None, None) == 1
    assert lib.attn_merge(FAKE, FAKE, FAKE, 2, 1, 1, 1, 80, FAKE, 0, None, None) == 2
    assert lib.attn_merge(FAKE, FAKE, FAKE, 2, 0, 1, 1, 64, FAKE, 0, None, None) == 0
    ws = lib.attn_jagged_workspace_bytes(3, 1000, 600)
    # counts, items, 3 units (padded to 16 bytes), then the worklist builder's table of
    # 64 int2 per started block of 1024 sequences
    assert ws == 16 + 16 * ((1000 + 3 * 127) // 128) + 32 + 512
    assert lib.attn_jagged_workspace_bytes(3000, 10 ** 6, 1024) == \
        16 + 16 * ((10 ** 6 + 3000 * 127) // 128) + 3000 * 8 + 3 * 512
    assert lib.attn_jagged(FAKE, FAKE, FAKE, FAKE, None, FAKE, 3, 1000, 600, 4, 128, 1, 0.1, 1, FAKE, ws - 1,
                           None) == 1
    assert lib.attn_jagged(FAKE, FAKE, FAKE, FAKE, None, None, 3, 1000, 600, 4, 128, 1, 0.1, 1, FAKE, ws,
                           None) == 1
    assert lib.attn_jagged(FAKE, FAKE, FAKE, FAKE, None, FAKE, 0, 1000, 600, 4, 128, 1, 0.1, 1, FAKE, ws,
                           None) == 0
    wd = lib.attn_decode_workspace_bytes(8, 64, 128, 64)
    # m, l (16-byte aligned), O partials, then B * h_q int32 merge counters (16-byte aligned)
    assert wd == ((64 * 8 * 64 * 2 * 4 + 15) // 16) * 16 + 64 * 8 * 64 * 128 * 4 + ((8 * 64 * 4 + 15) // 16) * 16
    assert lib.attn_decode_splitkv(FAKE, FAKE, FAKE, FAKE, None, 8, 1000, 64, 2, 128, 1, 0.1, 4, FAKE, wd,
                                   None) == 2  # G = 32 > 16
    assert lib.attn_decode_splitkv(FAKE, FAKE, FAKE, FAKE, None, 8, 1000, 64, 8, 128, 1, 0.1, 0, FAKE, wd,
                                   None) == 1
    assert lib.attn_decode_splitkv(FAKE, FAKE, FAKE, FAKE, None, 8, 1000, 64, 8, 128, 1, 0.1, 64, FAKE, 16,
                                   None) == 1


def test_probe_validation(lib):
    assert lib.attn_probe_mma_cycles(None, 16, None) == 1
    assert lib.attn_probe_mma_cycles(ctypes.c_void_p(0x10004), 16, None) == 1  # not 8-byte aligned
    assert lib.attn_probe_mma_cycles(FAKE, 0, None) == 1
    assert lib.attn_probe_mma_cycles(FAKE, (1 << 20) + 1, None) == 1


def test_status_strings(lib):
    for code in range(6):
        assert ra.attn_status_string(code) != "unknown status"
    assert ra.attn_status_string(99) == "unknown status"


def _walk_pairs(lo, hi, S_kv, causal, C, q_pos0=0, kv_pos0=0):
    lib_walk = ra.attn_tile_walk(lo, hi, 0, S_kv, block_n=128, causal=causal, num_chunks=C, q_pos0=q_pos0,
                                 kv_pos0=kv_pos0)
    ref = S.tile_walk(lo, hi, 0, S_kv, 128, causal, C, q_pos0, kv_pos0)
    return lib_walk, ref


@pytest.mark.parametrize("seed", range(60))
def test_tile_walk_matches_oracle_bit_exact(lib, seed):
    rng = np.random.default_rng(seed)
    S_q = int(rng.integers(1, 900))
    S_kv = S_q if rng.random() < 0.6 else int(rng.integers(0, 900))
    causal = bool(rng.random() < 0.7)
    C = int(rng.integers(1, 9))
    q_pos0 = int(rng.integers(-300, 300)) if rng.random() < 0.3 else 0
    for lo, hi in S.dense_work_items(S_q, 128):
        got, ref = _walk_pairs(lo, hi, S_kv, causal, C, q_pos0)
        assert [(c, s) for c, s, _ in got] == [(c, s) for c, s, _ in ref]
        chunks, _ = S.ring_chunks(0, S_kv, C)
        for (c, s, mend), (_, _, stop) in zip(got, ref):
            # the tail mask stops at the chunk end or earlier and never cuts a visible key
            assert mend <= chunks[c][1]
            if mend < stop:
                assert not S.pair_visible_in(lo, hi, mend, stop, causal, q_pos0, 0)


@pytest.mark.parametrize("seed", range(40))
def test_window_tile_walk_matches_oracle_bit_exact(lib, seed):
    """Sliding window: the library's walk starts at the grid tile holding the first
    visible key and keeps exactly the tiles that hold a visible (query, key) pair."""
    rng = np.random.default_rng(1000 + seed)
    L = int(rng.integers(1, 1200))
    C = int(rng.integers(1, 6))
    window = int(rng.choice([0, 1, 63, 127, 128, 129, 255, 300, 1000, 5000]))
    q_pos0 = int(rng.integers(-200, 200)) if rng.random() < 0.3 else 0
    for lo, hi in S.dense_work_items(L, 128):
        got = ra.attn_tile_walk(lo, hi, 0, L, block_n=128, causal=True, num_chunks=C, q_pos0=q_pos0, window=window)
        ref = S.tile_walk(lo, hi, 0, L, 128, True, C, q_pos0, 0, window)
        assert [(c, st) for c, st, _ in got] == [(c, st) for c, st, _ in ref]


@pytest.mark.parametrize("seed", range(60))
def test_tile_walk_aligned_ring_is_the_rotated_linear_walk(lib, seed):
    """Ring chunks whose length is a multiple of the 128-key tile: the library walks
    them as its single-chunk walk rotated to start at the Q tile's own chunk.  The
    tiles, their chunks and their order must equal the oracle's ring walk, with or
    without causal masking, a sliding window and position offsets."""
    rng = np.random.default_rng(1000 + seed)
    C = int(rng.integers(2, 9))
    L = 128 * int(rng.integers(1, 5))
    S_kv = int(rng.integers((L - 1) * C + 1, L * C + 1))  # ceil(S_kv / C) == L
    assert -(-S_kv // C) == L
    S_q = S_kv if rng.random() < 0.6 else int(rng.integers(1, S_kv + 300))
    causal = bool(rng.random() < 0.7)
    window = int(rng.choice([0, 100, 128, 300, 1000])) if causal and rng.random() < 0.4 else -1
    q_pos0 = int(rng.integers(-300, 300)) if rng.random() < 0.3 else 0
    for lo, hi in S.dense_work_items(S_q, 128):
        got = ra.attn_tile_walk(lo, hi, 0, S_kv, block_n=128, causal=causal, num_chunks=C, q_pos0=q_pos0,
                                window=window)
        ref = S.tile_walk(lo, hi, 0, S_kv, 128, causal, C, q_pos0, 0, None if window < 0 else window)
        assert len(ref) > 0 or not causal or window >= 0 or q_pos0 < 0
        assert [(c, st) for c, st, _ in got] == [(c, st) for c, st, _ in ref]
        chunks, _ = S.ring_chunks(0, S_kv, C)
        for (c, st, mend), (_, _, stop) in zip(got, ref):
            assert mend <= chunks[c][1]
            if mend < stop:
                assert not S.pair_visible_in(lo, hi, mend, stop, causal, q_pos0, 0)


def test_tile_walk_aligned_ring_edges(lib):
    """Rings of whole-tile chunks at their edges: a Q tile that sees nothing (queries
    before every key), one whose own chunk is the last and shorter than the rest, one
    that sees only its diagonal tile under a zero window, and a non-causal tile, which
    visits every tile starting from its own chunk."""
    assert ra.attn_tile_walk(0, 128, 0, 1024, causal=True, num_chunks=4, q_pos0=-500) == []
    # 1017 keys in 8 chunks of 128: the last chunk holds 121 keys
    w = ra.attn_tile_walk(896, 1017, 0, 1017, causal=True, num_chunks=8)
    assert [(c, st) for c, st, _ in w] == [(7, 896)] + [(c, 128 * c) for c in range(7)]
    assert w[0][2] == 1017  # the tail tile stops at the range's end
    assert all(me == 128 * (c + 1) for c, _, me in w[1:])
    assert ra.attn_tile_walk(512, 640, 0, 1024, causal=True, num_chunks=4, window=0) == [(2, 512, 640)]
    w = ra.attn_tile_walk(300, 428, 0, 1024, causal=False, num_chunks=4)
    assert [st for _, st, _ in w] == [256, 384, 512, 640, 768, 896, 0, 128]


def test_window_validation(lib):
    n = ctypes.c_int(0)
    assert lib.attn_tile_walk(0, 128, 0, 512, 128, 0, 1, 0, 0, 5, None, None, None, 0, ctypes.byref(n)) == 1  # window needs causal
    assert lib.attn_tile_walk(0, 128, 0, 512, 128, 1, 1, 0, 0, -2, None, None, None, 0, ctypes.byref(n)) == 1
    args = [FAKE, FAKE, FAKE, FAKE, None, 1, 128, 128, 2, 1, 128, 1, 0.1, -1, 1, None]
    assert lib.attn_prefill_window(*args) == 1  # negative window
    args[13] = 0
    args[10] = 96
    assert lib.attn_prefill_window(*args) == 2  # D outside {64,128,256}


def test_tile_walk_full_size_counts(lib):
    # dense causal S=4096: 528 tiles per (batch, head); ring S=32768, C=8: 32896 tiles
    tot = sum(len(ra.attn_tile_walk(lo, hi, 0, 4096, causal=True)) for lo, hi in S.dense_work_items(4096, 128))
    assert tot == 528
    tot = 0
    for lo, hi in S.dense_work_items(32768, 128):
        w = ra.attn_tile_walk(lo, hi, 0, 32768, causal=True, num_chunks=8)
        assert w[0][0] == lo // 4096  # starts on its own chunk
        tot += len(w)
    assert tot == 32896


def test_tile_walk_golden(lib, golden):
    for case in golden["schedule"]:
        if "walk" in case:
            lo, hi = case["q_tile"]
            got = ra.attn_tile_walk(lo, hi, 0, case["S"], causal=case["causal"], num_chunks=case["num_chunks"])
            assert [[c, s, min(s + 128, me)] for c, s, me in got] == case["walk"], case["name"]
