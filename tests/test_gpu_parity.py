"""GPU parity: every entry point against the fp64 oracle, element by element.

Tolerance (fixed for fp16/bf16 inputs, fp32 accumulation): max |O - O_ref| <= 1e-2,
mean |O - O_ref| <= 1e-3, |LSE - LSE_ref| <= 1e-3; -inf LSE and empty rows must
match exactly; integer outputs (worklists) bit-exact.
"""

import math

import numpy as np
import pytest
import torch

import ring_attention_online_gb300 as ra
import synthetic as syn
from oracle import attention as A
from oracle import schedule as S

pytestmark = pytest.mark.gpu

TOL_MAX, TOL_MEAN, TOL_LSE = 1e-2, 1e-3, 1e-3
DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ra.load_library()
    yield
    assert ra.attn_last_device_status() == 0


def close_o(got, ref, what=""):
    g = got.detach().float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.isfinite(g).all(), what
    err = np.abs(g - ref)
    assert err.max() <= TOL_MAX, f"{what}: max err {err.max():.3e}"
    assert err.mean() <= TOL_MEAN, f"{what}: mean err {err.mean():.3e}"


def close_lse(got, ref, what=""):
    g = got.detach().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    neg = np.isneginf(ref)
    assert np.array_equal(np.isneginf(g), neg), what
    if (~neg).any():
        err = np.abs(g[~neg] - ref[~neg])
        assert err.max() <= TOL_LSE, f"{what}: LSE err {err.max():.3e}"


def gen(shape_q, shape_kv, dtype, seed):
    return syn.qkv(shape_q, shape_kv, dtype, seed, "cuda")


# ---------------------------------------------------------------------- prefill
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S_,h_q,h_kv", [(300, 4, 2), (300, 2, 2), (520, 3, 1)])
def test_prefill_dense_ragged(D, dtype, causal, S_, h_q, h_kv):
    B = 2
    q, k, v = gen((B, S_, h_q, D), (B, S_, h_kv, D), dtype, seed=D + causal)
    o = torch.empty_like(q)
    lse = torch.empty(B, h_q, S_, device="cuda", dtype=torch.float32)
    scale = 1 / math.sqrt(D)
    ra.attn_prefill(q, k, v, o, lse, scale=scale, causal=causal)
    O, L = A.attention(q.cpu(), k.cpu(), v.cpu(), scale, causal)
    close_o(o, O, f"prefill D={D} {dtype} causal={causal}")
    close_lse(lse, L)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("C", [2, 3, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_prefill_ring_gqa(C, causal, dtype):
    """attn_prefill, general ring walk (1000 / C keys per chunk is not a whole number of
    128-key tiles), GQA head pairs, both input types."""
    B, S_, h_q, h_kv, D = 1, 1000, 8, 2, 128
    q, k, v = gen((B, S_, h_q, D), (B, S_, h_kv, D), dtype, seed=10 + C)
    o = torch.empty_like(q)
    lse = torch.empty(B, h_q, S_, device="cuda", dtype=torch.float32)
    ra.attn_prefill(q, k, v, o, lse, causal=causal, num_chunks=C)
    O, L = A.attention(q.cpu(), k.cpu(), v.cpu(), 1 / math.sqrt(D), causal)
    close_o(o, O, f"attn_prefill ring C={C} {dtype}")
    close_lse(lse, L)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S_,C,h_q,h_kv", [(1024, 4, 8, 2), (2048, 8, 4, 4), (1152, 3, 2, 2), (1100, 3, 6, 3)])
def test_prefill_ring_chunks_of_whole_tiles(D, causal, S_, C, h_q, h_kv, dtype):
    """Ring chunks whose length is a multiple of 128 keys (256, 384; 1100 / 3 -> 367 is
    not, for contrast) run as the single-chunk walk rotated to each Q tile's own chunk:
    head pairs and Q-tile pairs, 256-row items that straddle a chunk boundary (384-key
    chunks), causal and not."""
    B = 1
    q, k, v = gen((B, S_, h_q, D), (B, S_, h_kv, D), dtype, seed=90 + C + D)
    o = torch.empty_like(q)
    lse = torch.empty(B, h_q, S_, device="cuda", dtype=torch.float32)
    ra.attn_prefill(q, k, v, o, lse, causal=causal, num_chunks=C)
    O, L = A.attention(q.cpu(), k.cpu(), v.cpu(), 1 / math.sqrt(D), causal)
    close_o(o, O, f"attn_prefill ring of whole tiles S={S_} C={C} D={D} {dtype}")
    close_lse(lse, L)


@pytest.mark.parametrize("window", [0, 300, 700])
def test_prefill_window_ring_chunks_of_whole_tiles(window):
    B, S_, h_q, h_kv, D, C = 1, 2048, 8, 2, 128, 4
    q, k, v = gen((B, S_, h_q, D), (B, S_, h_kv, D), "bf16", seed=95 + window)
    o = torch.empty_like(q)
    lse = torch.empty(B, h_q, S_, device="cuda", dtype=torch.float32)
    ra.attn_prefill_window(q, k, v, o, lse, window=window, num_chunks=C)
    O, L = A.attention(q.cpu(), k.cpu(), v.cpu(), 1 / math.sqrt(D), True, window=window)
    close_o(o, O, f"window ring of whole tiles w={window}")
    close_lse(lse, L)


@pytest.mark.parametrize("C", [2, 3])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("h_q,h_kv", [(3, 3), (4, 2)])
def test_prefill_ring_d256_cta_pairs(C, causal, h_q, h_kv):
    """Head dim 256 (CTA pairs) with a ring walk over C chunks of 347 and 232 keys, not
    whole tiles: Q-tile pairs (MHA, the odd tile count leaves rank 1 an empty tile) and
    head pairs (even GQA group), causal and full."""
    B, S_, D = 2, 694, 256
    q, k, v = gen((B, S_, h_q, D), (B, S_, h_kv, D), "bf16", seed=120 + C + h_q)
    o = torch.empty_like(q)
    lse = torch.empty(B, h_q, S_, device="cuda", dtype=torch.float32)
    ra.attn_prefill(q, k, v, o, lse, causal=causal, num_chunks=C)
    O, L = A.attention(q.cpu(), k.cpu(), v.cpu(), 1 / math.sqrt(D), causal)
    close_o(o, O, f"attn_prefill D=256 ring C={C} causal={causal} heads {h_q}/{h_kv}")
    close_lse(lse, L)


@pytest.mark.parametrize("window", [100, 300])
def test_prefill_window_ring_d256_cta_pairs(window):
    """Head dim 256 sliding window over a three-chunk ring (a pair's rows at the lower
    window edge see fewer tiles than the pair walks)."""
    B, S_, h_q, h_kv, D = 1, 900, 4, 4, 256
    q, k, v = gen((B, S_, h_q, D), (B, S_, h_kv, D), "fp16", seed=130 + window)
    o = torch.empty_like(q)
    lse = torch.empty(B, h_q, S_, device="cuda", dtype=torch.float32)
    ra.attn_prefill_window(q, k, v, o, lse, window=window, num_chunks=3)
    O, L = A.attention(q.cpu(), k.cpu(), v.cpu(), 1 / math.sqrt(D), True, window=window)
    close_o(o, O, f"attn_prefill_window D=256 ring w={window}")
    close_lse(lse, L)


# ---------------------------------------------------------------------- sliding window
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("window", [0, 1, 100, 127, 128, 129, 300, 5000])
@pytest.mark.parametrize("h_q,h_kv", [(4, 2), (2, 2)])
def test_prefill_window_parity(D, window, h_q, h_kv, dtype):
    """Both kernels (paired for 64/128 with head pairs and Q-tile pairs, CTA pairs for
    256): the walk floor, the per-row lower mask and sub-tiles sitting out tiles below
    their window; window 5000 > S is plain causal."""
    B, S_ = 1, 650
    q, k, v = gen((B, S_, h_q, D), (B, S_, h_kv, D), dtype, seed=window + D)
    o = torch.empty_like(q)
    lse = torch.empty(B, h_q, S_, device="cuda", dtype=torch.float32)
    scale = 1 / math.sqrt(D)
    ra.attn_prefill_window(q, k, v, o, lse, window=window, scale=scale)
    O, L = A.attention(q.cpu(), k.cpu(), v.cpu(), scale, True, window=window)
    close_o(o, O, f"attn_prefill_window window={window} D={D} {dtype}")
    close_lse(lse, L)


@pytest.mark.parametrize("C", [1, 3, 8])
def test_prefill_window_ring_gqa(C):
    B, S_, h_q, h_kv, D, window = 1, 2000, 8, 2, 128, 700
    q, k, v = gen((B, S_, h_q, D), (B, S_, h_kv, D), "bf16", seed=40 + C)
    o = torch.empty_like(q)
    lse = torch.empty(B, h_q, S_, device="cuda", dtype=torch.float32)
    ra.attn_prefill_window(q, k, v, o, lse, window=window, num_chunks=C)
    O, L = A.attention(q.cpu(), k.cpu(), v.cpu(), 1 / math.sqrt(D), True, window=window)
    close_o(o, O, f"window ring C={C}")
    close_lse(lse, L)


# ---------------------------------------------------------------------- persistent grids
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_d256_persistent_many_units(causal):
    """Head dim 256 runs one CTA pair per two SMs over units of two 256-row pair items;
    with an even group size (48 / 8 = 6) an item is one Q tile of two query heads.  Here
    there are more than twice as many units as pairs, so every pair chains several, and
    the odd Q-tile count gives every (batch, head pair) a unit with an empty second slot
    (the causal middle tile, the non-causal last one)."""
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    B, S_, h_q, h_kv, D = 4, 300, 48, 8, 256
    n_it = (S_ + 127) // 128  # pair items per (batch, head pair)
    units = B * (h_q // 2) * ((n_it + 1) // 2)
    assert units > 2 * pairs
    q, k, v = gen((B, S_, h_q, D), (B, S_, h_kv, D), "bf16", seed=60 + causal)
    o = torch.empty_like(q)
    lse = torch.empty(B, h_q, S_, device="cuda", dtype=torch.float32)
    ra.attn_prefill(q, k, v, o, lse, causal=causal)
    O, L = A.attention(q.cpu(), k.cpu(), v.cpu(), 1 / math.sqrt(D), causal)
    close_o(o, O, f"persistent D=256 causal={causal}")
    close_lse(lse, L)


@pytest.mark.parametrize("C", [1, 3])
@pytest.mark.parametrize("D,h_q,h_kv", [(128, 16, 8), (64, 12, 12)])
def test_prefill_window_persistent_many_items(D, h_q, h_kv, C):
    """Sliding-window launches of the paired kernel are persistent (items in a snake
    order over one CTA per SM): more items than SMs, as head pairs (GQA) and as Q-tile
    pairs, with a ragged last tile, in one chunk and in a three-chunk ring walk."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, S_, window = 3, 1100, 300
    rows = 128 if (h_q // h_kv) % 2 == 0 else 256
    items = B * ((S_ + rows - 1) // rows) * (h_q // 2 if rows == 128 else h_q)
    assert items > sms
    q, k, v = gen((B, S_, h_q, D), (B, S_, h_kv, D), "bf16", seed=70 + D)
    o = torch.empty_like(q)
    lse = torch.empty(B, h_q, S_, device="cuda", dtype=torch.float32)
    ra.attn_prefill_window(q, k, v, o, lse, window=window, num_chunks=C)
    O, L = A.attention(q.cpu(), k.cpu(), v.cpu(), 1 / math.sqrt(D), True, window=window)
    close_o(o, O, f"persistent window D={D} C={C}")
    close_lse(lse, L)


@pytest.mark.parametrize("S_q,S_kv", [(200, 700), (700, 200), (1, 513), (129, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_prefill_unequal_lengths(S_q, S_kv, causal):
    q, k, v = gen((1, S_q, 2, 64), (1, S_kv, 1, 64), "bf16", seed=S_q)
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, S_q, device="cuda", dtype=torch.float32)
    ra.attn_prefill(q, k, v, o, lse, causal=causal, num_chunks=2)
    O, L = A.attention(q.cpu(), k.cpu(), v.cpu(), 1 / 8, causal)
    close_o(o, O)
    close_lse(lse, L)


@pytest.mark.parametrize("D,S_q", [(64, 130), (128, 300), (256, 300), (256, 130)])
@pytest.mark.parametrize("causal", [0, 1])
def test_prefill_empty_kv_gives_zero_and_neg_inf(D, S_q, causal):
    """No keys: O = 0 and LSE = -inf for every row.  At head dim 256 a CTA takes two Q
    tiles in turn (S_q = 300: three tiles, one CTA with two empty items)."""
    q, _, _ = gen((1, S_q, 2, D), (1, 1, 2, D), "bf16", seed=3)
    k = torch.empty(1, 1, 2, D, device="cuda", dtype=torch.bfloat16)  # any valid pointer
    o = torch.full_like(q, 7.0)
    lse = torch.zeros(1, 2, S_q, device="cuda")
    lib = ra.load_library()
    import ctypes
    st = lib.attn_prefill(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                          ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()), 1, S_q, 0, 2, 2, D, 1,
                          1 / math.sqrt(D), causal, 1, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert ra.attn_last_device_status() == 0
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


# ---------------------------------------------------------------------- partial + merge
def test_tiny_config_partials_merge_and_ring():
    """B=1, h_q=2, h_kv=1, S=256, D=64, fp16, non-causal, C=4 chunks of 64 keys."""
    cfg = syn.WORKLOADS["tiny_gqa_ring4"]
    q, k, v = syn.prefill_inputs(cfg, seed=0, device="cuda")
    B, S_, h_q, D, C = cfg["B"], cfg["S_q"], cfg["h_q"], cfg["D"], cfg["num_chunks"]
    scale = 1 / math.sqrt(D)
    m = torch.empty(C, B, h_q, S_, device="cuda")
    l = torch.empty_like(m)
    o_un = torch.empty(C, B, S_, h_q, D, device="cuda")
    for c in range(C):
        ra.attn_partial(q, k, v, m[c], l[c], o_un[c], scale=scale, causal=False, kv_begin=64 * c, kv_end=64 * (c + 1))
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    for c in range(C):
        mr, lr, orr = A.partial(qc, kc, vc, scale, False, 0, 64 * c, 64 * (c + 1))
        assert np.abs(m[c].cpu().numpy() - mr).max() <= 1e-3
        assert np.abs(l[c].cpu().numpy() / lr - 1).max() <= 1e-3
        close_o(o_un[c] / l[c].permute(0, 2, 1)[..., None], orr / np.swapaxes(lr, 1, 2)[..., None], f"partial {c}")
    out = torch.empty_like(q)
    lse = torch.empty(B, h_q, S_, device="cuda")
    ra.attn_merge(m, l, o_un, out, lse)
    O, L = A.attention(qc, kc, vc, scale, False)
    close_o(out, O, "merge")
    close_lse(lse, L)
    o2 = torch.empty_like(q)
    lse2 = torch.empty_like(lse)
    ra.attn_prefill(q, k, v, o2, lse2, scale=scale, causal=False, num_chunks=C)
    close_o(o2, O, "ring prefill")
    close_lse(lse2, L)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_partial_causal_positions_and_identity(D, dtype):
    """attn_partial with causal positions (q_pos0), a range that nothing sees and an empty range."""
    B, S_q, S_kv, h = 1, 160, 600, 2
    q, k, v = gen((B, S_q, h, D), (B, S_kv, h, D), dtype, seed=D)
    scale = 1 / math.sqrt(D)
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    # queries at positions 300..459 against keys [250, 520): partly visible, row by row
    m = torch.empty(B, h, S_q, device="cuda")
    l = torch.empty_like(m)
    o = torch.empty(B, S_q, h, D, device="cuda")
    ra.attn_partial(q, k, v, m, l, o, scale=scale, causal=True, q_pos0=300, kv_begin=250, kv_end=520)
    mr, lr, orr = A.partial(qc, kc, vc, scale, True, 300, 250, 520)
    assert np.abs(m.cpu().numpy() - mr).max() <= 1e-3
    assert np.abs(l.cpu().numpy() / lr - 1).max() <= 1e-3
    close_o(o / l.permute(0, 2, 1)[..., None], orr / np.swapaxes(lr, 1, 2)[..., None], f"attn_partial D={D} {dtype}")
    # queries at positions 0..159 against keys [400, 600): nothing visible -> identity
    ra.attn_partial(q, k, v, m, l, o, scale=scale, causal=True, q_pos0=0, kv_begin=400, kv_end=600)
    torch.cuda.synchronize()
    assert torch.all(torch.isneginf(m)) and torch.all(l == 0) and torch.all(o == 0)
    # empty range -> identity
    ra.attn_partial(q, k, v, m, l, o, scale=scale, causal=False, kv_begin=17, kv_end=17)
    torch.cuda.synchronize()
    assert torch.all(torch.isneginf(m)) and torch.all(l == 0) and torch.all(o == 0)


def test_partial_d256_persistent_many_units():
    """Partials at head dim 256 run on the persistent grid of CTA pairs: more units
    than pairs, GQA (head-pair items), causal positions that leave some Q tiles fully
    visible, some partly and some (the earliest rows) with no visible key at all, so
    that empty items and identity rows sit between full ones in a pair's sequence of
    units."""
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    B, S_q, S_kv, h_q, h_kv, D = 3, 520, 900, 48, 8, 256
    assert B * (h_q // 2) * (((S_q + 127) // 128 + 1) // 2) > pairs
    q, k, v = gen((B, S_q, h_q, D), (B, S_kv, h_kv, D), "bf16", seed=81)
    scale = 1 / math.sqrt(D)
    m = torch.empty(B, h_q, S_q, device="cuda")
    l = torch.empty_like(m)
    o = torch.empty(B, S_q, h_q, D, device="cuda")
    # queries at positions 200..719 against keys [300, 800)
    ra.attn_partial(q, k, v, m, l, o, scale=scale, causal=True, q_pos0=200, kv_begin=300, kv_end=800)
    mr, lr, orr = A.partial(q.cpu(), k.cpu(), v.cpu(), scale, True, 200, 300, 800)
    mg, lg = m.cpu().numpy(), l.cpu().numpy()
    empty = np.isneginf(mr)
    assert empty.any() and (~empty).any()
    assert np.array_equal(np.isneginf(mg), empty)
    assert np.all(lg[empty] == 0)
    assert np.abs(mg[~empty] - mr[~empty]).max() <= 1e-3
    assert np.abs(lg[~empty] / lr[~empty] - 1).max() <= 1e-3
    full = ~np.swapaxes(empty, 1, 2)  # [B, S_q, h_q]
    og = (o / l.clamp_min(1e-30).permute(0, 2, 1)[..., None]).cpu().numpy()
    ref = orr / np.where(lr > 0, lr, 1.0).swapaxes(1, 2)[..., None]
    close_o(torch.from_numpy(og[full]), ref[full], "partial D=256 persistent")
    assert np.all(o.cpu().numpy()[~full] == 0)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D", [128, 256])
def test_merge_with_empty_partials_matches_full(D, dtype):
    """attn_partial over five causal ranges (two empty) then attn_merge into the input type."""
    B, S_, h = 2, 70, 3
    q, k, v = gen((B, S_, h, D), (B, S_, h, D), dtype, seed=5 + D)
    scale = 1 / math.sqrt(D)
    bounds = [(0, 10), (10, 10), (10, 69), (69, 70), (70, 70)]
    C = len(bounds)
    m = torch.empty(C, B, h, S_, device="cuda")
    l = torch.empty_like(m)
    o_un = torch.empty(C, B, S_, h, D, device="cuda")
    for c, (lo, hi) in enumerate(bounds):
        ra.attn_partial(q, k, v, m[c], l[c], o_un[c], scale=scale, causal=True, kv_begin=lo, kv_end=hi)
    out = torch.empty_like(q)
    lse = torch.empty(B, h, S_, device="cuda")
    ra.attn_merge(m, l, o_un, out, lse)
    O, L = A.attention(q.cpu(), k.cpu(), v.cpu(), scale, True)
    close_o(out, O, f"attn_merge D={D} {dtype}")
    close_lse(lse, L)


# ---------------------------------------------------------------------- jagged
def _jagged_case(lengths, H, D, seed, causal=True, dtype="bf16"):
    offs = syn.offsets_from_lengths(lengths)
    T = int(offs[-1])
    q, k, v = syn.qkv((T, H, D), (T, H, D), dtype, seed, "cuda")
    o = torch.empty_like(q)
    lse = torch.empty(H, T, device="cuda")
    max_len = int(max(lengths)) if len(lengths) else 0
    ws = torch.empty(ra.attn_jagged_workspace_bytes(len(lengths), T, max_len), dtype=torch.uint8, device="cuda")
    offs_d = torch.from_numpy(offs).cuda()
    ra.attn_jagged(q, k, v, o, offs_d, max_len, ws, lse, causal=causal)
    return q, k, v, o, lse, offs, ws


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [True, False])
def test_jagged_parity_and_worklist(causal, D, dtype):
    """attn_jagged: zero-length, 1-token and 127/128/129-token sequences, both input types."""
    lengths = [0, 1, 5, 127, 128, 129, 300, 1024, 77, 0, 256, 640, 383, 384, 385]
    H = 2
    q, k, v, o, lse, offs, ws = _jagged_case(lengths, H, D, seed=21, causal=causal, dtype=dtype)
    O, L = A.jagged_attention(q.cpu(), k.cpu(), v.cpu(), offs, 1 / math.sqrt(D), causal)
    close_o(o, O, f"attn_jagged D={D} causal={causal} {dtype}")
    close_lse(lse, L)
    _check_worklist(ws, offs, lengths, causal)


def _check_worklist(ws, offs, lengths, causal):
    """The device worklist in `ws` against the oracle's flattened worklist, bit for bit.
    Every head dim runs two 128-row sub-tiles per item (head dims 64/128 in one CTA,
    256 on a CTA pair), so the Q tiles are 256 rows."""
    block_m = 256
    words = ws.view(torch.int32).cpu().numpy()
    count = int(words[0])
    items = words[4:4 + 4 * count].reshape(count, 4)
    ref = S.jagged_worklist(offs, block_m, 128, causal)
    assert count == len(ref)
    got = sorted(map(tuple, items.tolist()))
    want = sorted((it["ordered_begin"], it["range_len"], it["tile_start"], it["tile_extent"]) for it in ref)
    assert got == want
    # order: non-increasing Q-tile count per sequence, and each sequence's tiles first-to-last
    ntiles = [(r[1] + block_m - 1) // block_m for r in items]
    assert all(a >= b for a, b in zip(ntiles, ntiles[1:]))
    # sequences of one tile count in index order (sequence starts ascend)
    for a, b in zip(items, items[1:]):
        if a[0] == b[0]:
            assert b[2] == a[2] + block_m
        elif (a[1] + block_m - 1) // block_m == (b[1] + block_m - 1) // block_m:
            assert a[0] < b[0]
    # units: one per non-empty sequence, covering its contiguous items in order
    n_units = int(words[1])
    max_items = (int(offs[-1]) + (len(offs) - 1) * (block_m - 1)) // block_m
    units = words[4 + 4 * max_items:4 + 4 * max_items + 2 * n_units].reshape(n_units, 2)
    assert n_units == sum(1 for n in lengths if n > 0)
    assert units[0][0] == 0 and all(u[1] >= 1 for u in units)
    for u, u2 in zip(units, units[1:]):
        assert u2[0] == u[0] + u[1]
    assert units[-1][0] + units[-1][1] == count
    for u in units:
        seq = items[u[0]:u[0] + u[1]]
        assert all(r[0] == seq[0][0] for r in seq) and u[1] == (seq[0][1] + block_m - 1) // block_m


@pytest.mark.parametrize("odd_high", [True, False])
def test_jagged_extreme_score_jumps(odd_high):
    """Keys in every other 128-key tile of a sequence score ~196 log2 units above the
    rest, so between consecutive KV tiles the running max jumps (or the tile adds only
    weights that underflow to zero in fp32): the online-softmax rescale factor is 0 and
    the lazily raised reference must still give the exact mean of the high keys' V.
    The lengths include lone last Q tiles and partial tiles of both parities."""
    lengths = [300, 640, 1100, 385, 1000]
    H, D = 2, 128
    offs = syn.offsets_from_lengths(lengths)
    T = int(offs[-1])
    q, k, v = syn.qkv((T, H, D), (T, H, D), "bf16", 31, "cuda")
    pos = torch.arange(T, device="cuda")
    rel = pos - torch.from_numpy(offs[:-1].astype(np.int64)).cuda().repeat_interleave(
        torch.tensor(lengths, device="cuda"))
    odd = ((rel // 128) % 2 == 1)[:, None, None]
    hi = odd if odd_high else ~odd
    q = (2.0 + 0.1 * q.float()).to(torch.bfloat16)
    k = torch.where(hi, 3.0 + 0.1 * k.float(), -3.0 + 0.1 * k.float()).to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(H, T, device="cuda")
    ws = torch.empty(ra.attn_jagged_workspace_bytes(len(lengths), T, max(lengths)), dtype=torch.uint8,
                     device="cuda")
    ra.attn_jagged(q, k, v, o, torch.from_numpy(offs).cuda(), max(lengths), ws, lse, causal=True)
    O, L = A.jagged_attention(q.cpu(), k.cpu(), v.cpu(), offs, 1 / math.sqrt(D), True)
    close_o(o, O)
    close_lse(lse, L)


@pytest.mark.parametrize("D", [64, 128])
def test_output_base_16_bytes_past_32(D):
    """The paired kernel stores O rows in 32-byte pieces when the output's base allows
    it and in 16-byte pieces otherwise: outputs 16 bytes past a 32-byte boundary."""
    B, S_, h = 1, 300, 2
    q, k, v = gen((B, S_, h, D), (B, S_, h, D), "bf16", seed=77)
    buf = torch.zeros(q.numel() + 16, dtype=q.dtype, device="cuda")
    o = buf[8:8 + q.numel()].view(q.shape)
    assert o.data_ptr() % 32 == 16
    lse = torch.empty(B, h, S_, device="cuda")
    ra.attn_prefill(q, k, v, o, lse, causal=True)
    O, L = A.attention(q.cpu(), k.cpu(), v.cpu(), 1 / math.sqrt(D), True)
    close_o(o, O, "dense, offset output")
    close_lse(lse, L)
    assert torch.all(buf[:8] == 0) and torch.all(buf[8 + q.numel():] == 0)
    lengths = [300, 77, 640]
    offs = syn.offsets_from_lengths(lengths)
    T = int(offs[-1])
    q, k, v = syn.qkv((T, h, D), (T, h, D), "bf16", 78, "cuda")
    buf = torch.zeros(q.numel() + 16, dtype=q.dtype, device="cuda")
    o = buf[8:8 + q.numel()].view(q.shape)
    lse = torch.empty(h, T, device="cuda")
    ws = torch.empty(ra.attn_jagged_workspace_bytes(len(lengths), T, 640), dtype=torch.uint8, device="cuda")
    ra.attn_jagged(q, k, v, o, torch.from_numpy(offs).cuda(), 640, ws, lse, causal=True)
    O, L = A.jagged_attention(q.cpu(), k.cpu(), v.cpu(), offs, 1 / math.sqrt(D), True)
    close_o(o, O, "jagged, offset output")
    close_lse(lse, L)
    assert torch.all(buf[:8] == 0) and torch.all(buf[8 + q.numel():] == 0)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_jagged_odd_tile_counts(D):
    """attn_jagged, causal: sequences of 1, 3, 5, 7 and 9 Q tiles of 128 rows (full and
    ragged last tiles) next to even counts.  A causal sequence with an odd tile count is
    cut into items {0}, {1, 2}, {3, 4}, ... (its first tile alone), the worklist's items
    into 256-row tiles from the start; every row must still come out once and right."""
    lengths = [128, 129, 255, 256, 257, 383, 384, 385, 511, 512, 640, 700, 768, 896, 897, 1024, 1100, 1152,
               1, 64, 130, 300, 520, 1000]
    H = 2
    q, k, v, o, lse, offs, _ = _jagged_case(lengths, H, D, seed=31 + D)
    O, L = A.jagged_attention(q.cpu(), k.cpu(), v.cpu(), offs, 1 / math.sqrt(D), True)
    close_o(o, O, f"attn_jagged odd tile counts D={D}")
    close_lse(lse, L)


def _sampled_jagged_parity(q, k, v, o, lse, offs, seqs, what):
    """Sequences `seqs` of a packed jagged batch against the oracle, one by one."""
    D = q.shape[-1]
    for b in seqs:
        lo, hi = int(offs[b]), int(offs[b + 1])
        if hi == lo:
            continue
        sl = slice(lo, hi)
        O, L = A.jagged_attention(q[sl].cpu(), k[sl].cpu(), v[sl].cpu(), np.array([0, hi - lo]), 1 / math.sqrt(D), True)
        close_o(o[sl], O, f"{what}, sequence {b}")
        close_lse(lse[:, sl], L)


def test_jagged_many_sequences_worklist():
    """More than 1024 sequences: the worklist is built by a count kernel and a write
    kernel over several CTAs.  5000 sequences of the jagged workload's lengths (64 to
    1024 tokens, so four tile-count buckets) with zero-length ones among them and
    sequences on the builder's CTA boundaries: the list bit for bit against the oracle's,
    and a seeded sample of sequences against the oracle."""
    rng = np.random.default_rng(41)
    lengths = rng.integers(64, 1025, 5000)
    lengths[rng.choice(5000, 50, replace=False)] = 0
    lengths[[0, 1023, 1024, 2047, 2048, 4999]] = [1024, 0, 513, 256, 64, 1000]
    q, k, v, o, lse, offs, ws = _jagged_case(lengths, 1, 64, seed=43)
    assert ra.attn_last_device_status() == 0
    _check_worklist(ws, offs, lengths, True)
    sample = sorted(set(rng.choice(5000, 60, replace=False).tolist()) | {0, 1023, 1024, 2047, 2048, 4999})
    _sampled_jagged_parity(q, k, v, o, lse, offs, sample, "attn_jagged 5000 sequences")


def test_jagged_many_sequences_unbucketed_order():
    """More than 1024 sequences with a longest one of more than 64 tiles of 256 rows:
    the worklist keeps sequence order (no tile-count buckets).  The list against the
    oracle's, and a seeded sample of sequences (the long one among them, checked on its
    first rows and sampled ones) against the oracle."""
    rng = np.random.default_rng(42)
    lengths = rng.integers(64, 1025, 1100)
    lengths[700] = 16500
    q, k, v, o, lse, offs, ws = _jagged_case(lengths, 1, 64, seed=44)
    assert ra.attn_last_device_status() == 0
    block_m = 256
    words = ws.view(torch.int32).cpu().numpy()
    count = int(words[0])
    items = words[4:4 + 4 * count].reshape(count, 4)
    ref = S.jagged_worklist(offs, block_m, 128, True)
    assert count == len(ref)
    assert sorted(map(tuple, items.tolist())) == sorted(
        (it["ordered_begin"], it["range_len"], it["tile_start"], it["tile_extent"]) for it in ref)
    # sequence order, each sequence's tiles first to last
    assert all(a[0] <= b[0] for a, b in zip(items, items[1:]))
    sample = sorted(set(rng.choice(1100, 40, replace=False).tolist()) - {700} | {0, 699, 701, 1099})
    _sampled_jagged_parity(q, k, v, o, lse, offs, sample, "attn_jagged 1100 sequences")
    # the long sequence: rows sampled across it, each against all the keys it sees
    lo = int(offs[700])
    rows = np.concatenate([np.arange(0, 300), np.sort(rng.choice(np.arange(300, 16500), 200, replace=False))])
    seq = slice(lo, lo + 16500)
    O, L = A.attention(q[None, seq].cpu(), k[None, seq].cpu(), v[None, seq].cpu(), 1 / 8, True, rows=rows)
    close_o(o[seq][rows], O[0, rows], "attn_jagged 16500-token sequence, sampled rows")
    close_lse(lse[:, seq][:, rows], L[0][:, rows])


def test_jagged_random_lengths():
    rng = np.random.default_rng(3)
    lengths = rng.integers(0, 700, 40)
    q, k, v, o, lse, offs, _ = _jagged_case(lengths, 4, 64, seed=22)
    O, L = A.jagged_attention(q.cpu(), k.cpu(), v.cpu(), offs, 1 / 8, True)
    close_o(o, O)
    close_lse(lse, L)


# ---------------------------------------------------------------------- decode
@pytest.mark.parametrize("D,h_q,h_kv,S_kv,splits", [
    (128, 16, 2, 5000, 7),     # G = 8, uneven splits, ragged tail
    (128, 16, 1, 4096, 64),    # G = 16
    (128, 4, 4, 777, 3),       # MHA, G = 1
    (64, 8, 1, 3000, 5),
    (256, 8, 2, 2000, 4),
    (128, 8, 1, 100, 16),      # more splits than 64-key tiles: empty chunks
])
def test_decode_parity_and_partials(D, h_q, h_kv, S_kv, splits):
    _decode_case(D, h_q, h_kv, S_kv, splits, "bf16")


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("G", [1, 8, 16])
def test_decode_fp16_parity_and_partials(D, G):
    """attn_decode_splitkv with fp16 inputs: the fused merge writes fp16 O; more splits
    than 64-key tiles (700 keys in 40 chunks of 18) leave the last chunk empty, an
    identity partial in the workspace."""
    h_kv = 2
    _decode_case(D, G * h_kv, h_kv, 700, 40, "fp16")


def _decode_case(D, h_q, h_kv, S_kv, splits, dtype):
    B = 2
    q, k, v = syn.qkv((B, h_q, D), (B, S_kv, h_kv, D), dtype, S_kv + D, "cuda")
    o = torch.empty_like(q)
    lse = torch.empty(B, h_q, device="cuda")
    ws = torch.empty(ra.attn_decode_workspace_bytes(B, h_q, D, splits), dtype=torch.uint8, device="cuda")
    scale = 1 / math.sqrt(D)
    ra.attn_decode_splitkv(q, k, v, o, ws, lse, num_splits=splits, scale=scale)
    assert o.dtype == q.dtype
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    O, L = A.decode(qc, kc, vc, scale, splits)
    close_o(o, O, f"attn_decode_splitkv D={D} G={h_q // h_kv} {dtype}")
    close_lse(lse, L)
    # the partial triplets in the documented workspace layout
    rows = splits * B * h_q
    f = ws.view(torch.float32)
    m = f[:rows].view(splits, B, h_q).cpu().numpy()
    l = f[rows:2 * rows].view(splits, B, h_q).cpu().numpy()
    off = ((rows * 8 + 15) // 16) * 4
    ou = f[off:off + rows * D].view(splits, B, h_q, D).cpu().numpy()
    mr, lr, orr = A.decode_partials(qc, kc, vc, scale, splits)
    empty = np.isneginf(mr)
    assert np.array_equal(np.isneginf(m), empty)
    assert np.all(l[empty] == 0) and np.all(ou[empty] == 0)
    assert np.abs(m[~empty] - mr[~empty]).max() <= 1e-3
    assert np.abs(l[~empty] / lr[~empty] - 1).max() <= 1e-3
    norm = ou[~empty] / l[~empty][:, None]
    ref_norm = orr[~empty] / lr[~empty][:, None]
    assert np.abs(norm - ref_norm).max() <= TOL_MAX


def test_decode_fused_merge_from_a_dirty_workspace_twice():
    """The group counters of the fused merge are zeroed by each call and left at zero."""
    B, h_q, h_kv, D, S_kv, splits = 3, 16, 2, 128, 3000, 9
    q, k, v = syn.qkv((B, h_q, D), (B, S_kv, h_kv, D), "bf16", 77, "cuda")
    scale = 1 / math.sqrt(D)
    nbytes = ra.attn_decode_workspace_bytes(B, h_q, D, splits)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")  # stale counters, NaN partials
    O, L = A.decode(q.cpu(), k.cpu(), v.cpu(), scale, splits)
    for _ in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, h_q), float("nan"), device="cuda")
        ra.attn_decode_splitkv(q, k, v, o, ws, lse, num_splits=splits, scale=scale)
        close_o(o, O)
        close_lse(lse, L)
    rows = splits * B * h_q
    off = ((rows * 8 + 15) // 16) * 16 + rows * D * 4
    counters = ws[off:off + B * h_kv * 4].view(torch.int32)
    assert (counters == 0).all()
    assert ra.attn_last_device_status() == 0


# ---------------------------------------------------------------------- failure detection
def test_bounded_wait_times_out_cleanly_and_context_survives():
    assert ra.attn_last_device_status() == 0
    ra.attn_selftest_wait_timeout(20_000_000)  # 20 ms
    assert ra.attn_last_device_status() == 4   # ATTN_ERR_TIMEOUT, reported once
    assert ra.attn_last_device_status() == 0
    q, k, v = gen((1, 64, 1, 64), (1, 64, 1, 64), "bf16", seed=1)
    o = torch.empty_like(q)
    ra.attn_prefill(q, k, v, o, causal=True)
    O, _ = A.attention(q.cpu(), k.cpu(), v.cpu(), 1 / 8, True)
    close_o(o, O)


def test_malformed_offsets_reported_as_device_input_error():
    offs = torch.tensor([0, 50, 30, 80], dtype=torch.int32, device="cuda")  # sequence 1 has negative length
    q = torch.randn(80, 1, 64, device="cuda").bfloat16()
    o = torch.zeros_like(q)
    ws = torch.empty(ra.attn_jagged_workspace_bytes(3, 80, 64), dtype=torch.uint8, device="cuda")
    ra.attn_jagged(q, q, q, o, offs, 64, ws)
    assert ra.attn_last_device_status() == 5
    assert ra.attn_last_device_status() == 0


# ---------------------------------------------------------------------- tensor-pipe probe
def test_probe_mma_rate_matches_the_nominal_per_sm_rate():
    """Back-to-back 128x128x16 bf16 MMAs on one SM issue every 64 cycles: 8192 FLOP per
    cycle per SM, the figure the nominal roofline denominator is built from."""
    cpm = ra.attn_probe_mma_cycles(2048)
    assert 60.0 <= cpm <= 72.0, cpm
    assert ra.attn_last_device_status() == 0
