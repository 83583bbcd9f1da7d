"""Pins of the fp64 oracle against things other than itself (CPU only).

Pins: a pure-Python brute force on tiny shapes, torch's scaled_dot_product_attention
in float64 (a library special case), hand-derived worked examples
(tests/golden/worked_examples.json), closed forms (zero queries give prefix means
and LSE = ln(i+1); a dominant key gives its value row), the merge identity and the
merge-equals-full-softmax theorem over arbitrary splits.
"""

import math

import numpy as np
import pytest
import torch

from oracle import attention as A

RNG = np.random.default_rng(1234)


# --------------------------------------------------------------------------
# brute force: scalar loops, no numpy arithmetic
# --------------------------------------------------------------------------
def brute_attention(q, k, v, scale, causal):
    B, S_q, h_q, D = q.shape
    S_kv, h_kv, Dv = k.shape[1], k.shape[2], v.shape[3]
    G = h_q // h_kv
    O = np.zeros((B, S_q, h_q, Dv))
    L = np.zeros((B, h_q, S_q))
    for b in range(B):
        for h in range(h_q):
            g = h // G
            for i in range(S_q):
                scores = []
                for j in range(S_kv):
                    if causal and j > i:
                        continue
                    s = 0.0
                    for d in range(D):
                        s += float(q[b, i, h, d]) * float(k[b, j, g, d])
                    scores.append((j, scale * s))
                mx = max(s for _, s in scores)
                den = sum(math.exp(s - mx) for _, s in scores)
                for e in range(Dv):
                    O[b, i, h, e] = sum(math.exp(s - mx) * float(v[b, j, g, e]) for j, s in scores) / den
                L[b, h, i] = mx + math.log(den)
    return O, L


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("h_q,h_kv", [(1, 1), (2, 1), (2, 2)])
def test_oracle_matches_brute_force(causal, h_q, h_kv):
    S, D = 13, 5
    q = RNG.standard_normal((1, S, h_q, D))
    k = RNG.standard_normal((1, S, h_kv, D))
    v = RNG.standard_normal((1, S, h_kv, D + 2))
    scale = 0.37
    O, L = A.attention(q, k, v, scale, causal)
    Ob, Lb = brute_attention(q, k, v, scale, causal)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, Lb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_oracle_matches_torch_sdpa_fp64(causal):
    B, S, h_q, h_kv, D = 2, 37, 4, 2, 16
    q = RNG.standard_normal((B, S, h_q, D))
    k = RNG.standard_normal((B, S, h_kv, D))
    v = RNG.standard_normal((B, S, h_kv, D))
    scale = 1 / math.sqrt(D)
    O, _ = A.attention(q, k, v, scale, causal)
    G = h_q // h_kv
    tq = torch.from_numpy(q).permute(0, 2, 1, 3)
    tk = torch.from_numpy(k).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    tv = torch.from_numpy(v).permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    np.testing.assert_allclose(O, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-10)


def test_golden_attention(golden):
    for case in golden["attention"]:
        O, L = A.attention(np.array(case["q"]), np.array(case["k"]), np.array(case["v"]),
                           case["scale"], case["causal"])
        np.testing.assert_allclose(O, np.array(case["O"]), rtol=0, atol=1e-14, err_msg=case["name"])
        np.testing.assert_allclose(L, np.array(case["LSE"]), rtol=0, atol=1e-14, err_msg=case["name"])


def test_golden_merge(golden):
    for case in golden["merge"]:
        m = np.array([float(x) for x in case["m"]]).reshape(-1, 1, 1, 1)
        l = np.array(case["l"], dtype=np.float64).reshape(-1, 1, 1, 1)
        o = np.array(case["O"], dtype=np.float64).reshape(-1, 1, 1, 1, len(case["O_final"]))
        O, L = A.merge(m, l, o)
        np.testing.assert_allclose(O.ravel(), case["O_final"], rtol=0, atol=1e-14, err_msg=case["name"])
        np.testing.assert_allclose(L.ravel(), [case["LSE"]], rtol=0, atol=1e-14, err_msg=case["name"])


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_closed_form(causal):
    """Q = 0: every visible key scores 0, so O_i = mean of the visible V rows and LSE_i = ln(#visible)."""
    B, S, h_q, h_kv, D = 2, 50, 4, 2, 8
    q = np.zeros((B, S, h_q, D))
    k = RNG.standard_normal((B, S, h_kv, D))
    v = RNG.standard_normal((B, S, h_kv, D))
    O, L = A.attention(q, k, v, 0.3, causal)
    G = h_q // h_kv
    for h in range(h_q):
        g = h // G
        if causal:
            expect = np.cumsum(v[:, :, g, :], axis=1) / np.arange(1, S + 1)[None, :, None]
            lse = np.log(np.arange(1, S + 1))
        else:
            expect = np.broadcast_to(v[:, :, g, :].mean(axis=1, keepdims=True), (B, S, D))
            lse = np.full(S, math.log(S))
        np.testing.assert_allclose(O[:, :, h, :], expect, rtol=0, atol=1e-12)
        np.testing.assert_allclose(L[:, h, :], np.broadcast_to(lse, (B, S)), rtol=0, atol=1e-12)


def test_dominant_key_returns_its_value():
    """One key aligned with q at a large margin: O ~ v_j to within e^-margin."""
    S, D = 20, 8
    q = RNG.standard_normal((1, S, 1, D))
    k = RNG.standard_normal((1, S, 1, D)) * 0.01
    j = 7
    k[0, j, 0] = 40.0 * q[0, 3, 0] / np.linalg.norm(q[0, 3, 0])
    v = RNG.standard_normal((1, S, 1, D))
    O, _ = A.attention(q, k, v, 1.0, False, rows=[3])
    margin = 40.0 * np.linalg.norm(q[0, 3, 0]) - 1.0
    assert np.abs(O[0, 3, 0] - v[0, j, 0]).max() < S * math.exp(-margin) * 10 + 1e-12


def test_fully_masked_rows_are_identity():
    """A row with no visible key: partial (-inf, 0, 0); normalised output O = 0, LSE = -inf."""
    q = RNG.standard_normal((1, 4, 1, 3))
    k = RNG.standard_normal((1, 8, 1, 3))
    v = RNG.standard_normal((1, 8, 1, 3))
    # queries at positions 0..3 see none of the keys 4..7 under causal masking
    m, l, o = A.partial(q, k, v, 1.0, True, q_pos0=0, kv_begin=4, kv_end=8)
    assert np.all(m == -np.inf) and np.all(l == 0) and np.all(o == 0)
    O, L = A.attention(q, k[:, 4:], v[:, 4:], 1.0, True, q_pos0=0, kv_pos0=4)
    assert np.all(O == 0) and np.all(L == -np.inf)


def _random_split(n, parts):
    cuts = np.sort(RNG.integers(0, n + 1, parts - 1))
    bounds = np.concatenate([[0], cuts, [n]])
    return [(int(bounds[i]), int(bounds[i + 1])) for i in range(parts)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("parts", [1, 2, 3, 7])
def test_merge_of_any_split_equals_full_softmax(causal, parts):
    B, S, h_q, h_kv, D = 1, 40, 2, 1, 6
    q = RNG.standard_normal((B, S, h_q, D))
    k = RNG.standard_normal((B, S, h_kv, D)) * 2
    v = RNG.standard_normal((B, S, h_kv, D))
    ranges = _random_split(S, parts) + [(5, 5)]  # plus an empty range
    trip = [A.partial(q, k, v, 0.7, causal, 0, lo, hi) for lo, hi in ranges]
    ms = np.stack([t[0] for t in trip])
    ls = np.stack([t[1] for t in trip])
    os_ = np.stack([t[2] for t in trip])
    O_ref, L_ref = A.attention(q, k, v, 0.7, causal)
    for order in (None, list(reversed(range(len(ranges)))), list(RNG.permutation(len(ranges)))):
        O, L = A.merge(ms, ls, os_, order)
        np.testing.assert_allclose(O, O_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(L, L_ref, rtol=0, atol=1e-12)


def test_injected_empty_partials_leave_merge_bit_identical():
    B, S, H, D = 1, 16, 2, 4
    q = RNG.standard_normal((B, S, H, D))
    k = RNG.standard_normal((B, S, H, D))
    v = RNG.standard_normal((B, S, H, D))
    parts = [A.partial(q, k, v, 0.5, False, 0, lo, hi) for lo, hi in [(0, 5), (5, 16)]]
    ms = np.stack([p[0] for p in parts])
    ls = np.stack([p[1] for p in parts])
    os_ = np.stack([p[2] for p in parts])
    O1, L1 = A.merge(ms, ls, os_)
    ident_m = np.full((1,) + ms.shape[1:], -np.inf)
    ident_l = np.zeros((1,) + ls.shape[1:])
    ident_o = np.zeros((1,) + os_.shape[1:])
    O2, L2 = A.merge(np.concatenate([ms[:1], ident_m, ms[1:], ident_m]),
                     np.concatenate([ls[:1], ident_l, ls[1:], ident_l]),
                     np.concatenate([os_[:1], ident_o, os_[1:], ident_o]))
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("C", [1, 3, 4])
def test_ring_prefill_equals_attention(causal, C):
    B, S, h_q, h_kv, D = 1, 48, 2, 1, 8
    q = RNG.standard_normal((B, S, h_q, D))
    k = RNG.standard_normal((B, S, h_kv, D))
    v = RNG.standard_normal((B, S, h_kv, D))
    O_ref, L_ref = A.attention(q, k, v, 0.35, causal)
    O, L = A.ring_prefill(q, k, v, 0.35, causal, C)
    np.testing.assert_allclose(O, O_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, L_ref, rtol=0, atol=1e-12)


def test_jagged_zero_query_prefix_means_per_segment():
    lens = [5, 0, 9, 1, 17]
    offs = np.concatenate([[0], np.cumsum(lens)])
    T, H, D = offs[-1], 2, 3
    q = np.zeros((T, H, D))
    k = RNG.standard_normal((T, H, D))
    v = RNG.standard_normal((T, H, D))
    O, L = A.jagged_attention(q, k, v, offs, 0.5, True)
    for b in range(len(lens)):
        lo, hi = offs[b], offs[b + 1]
        if hi == lo:
            continue
        n = np.arange(1, hi - lo + 1)
        np.testing.assert_allclose(O[lo:hi], np.cumsum(v[lo:hi], axis=0) / n[:, None, None], atol=1e-12)
        np.testing.assert_allclose(L[:, lo:hi], np.broadcast_to(np.log(n), (H, hi - lo)), atol=1e-12)


def test_jagged_matches_brute_force_per_sequence():
    lens = [3, 6, 1]
    offs = np.concatenate([[0], np.cumsum(lens)])
    T, H, D = offs[-1], 2, 4
    q = RNG.standard_normal((T, H, D))
    k = RNG.standard_normal((T, H, D))
    v = RNG.standard_normal((T, H, D))
    O, L = A.jagged_attention(q, k, v, offs, 0.6, True)
    for b in range(len(lens)):
        lo, hi = offs[b], offs[b + 1]
        Ob, Lb = brute_attention(q[None, lo:hi], k[None, lo:hi], v[None, lo:hi], 0.6, True)
        np.testing.assert_allclose(O[lo:hi], Ob[0], atol=1e-12)
        np.testing.assert_allclose(L[:, lo:hi], Lb[0], atol=1e-12)


@pytest.mark.parametrize("splits", [1, 4, 7])
def test_decode_equals_single_query_attention(splits):
    B, S, h_q, h_kv, D = 2, 45, 4, 2, 8
    q = RNG.standard_normal((B, h_q, D))
    k = RNG.standard_normal((B, S, h_kv, D))
    v = RNG.standard_normal((B, S, h_kv, D))
    O, L = A.decode(q, k, v, 0.3, splits)
    Ob, Lb = brute_attention(q[:, None], k, v, 0.3, False)
    np.testing.assert_allclose(O, Ob[:, 0], atol=1e-12)
    np.testing.assert_allclose(L, Lb[:, :, 0], atol=1e-12)


def test_decode_split_remainder_and_empty_chunks():
    """ceil-sized chunks: S=10 in 4 splits is 3,3,3,1; S=3 in 5 splits leaves empty chunks."""
    assert A.chunk_bounds(10, 4) == [(0, 3), (3, 6), (6, 9), (9, 10)]
    assert A.chunk_bounds(3, 5) == [(0, 1), (1, 2), (2, 3), (3, 3), (3, 3)]
    q = RNG.standard_normal((1, 2, 4))
    k = RNG.standard_normal((1, 3, 1, 4))
    v = RNG.standard_normal((1, 3, 1, 4))
    m, l, o = A.decode_partials(q, k, v, 1.0, 5)
    assert np.all(m[3:] == -np.inf) and np.all(l[3:] == 0) and np.all(o[3:] == 0)
    O, _ = A.decode(q, k, v, 1.0, 5)
    Ob, _ = brute_attention(q[:, None], k, v, 1.0, False)
    np.testing.assert_allclose(O, Ob[:, 0], atol=1e-12)


def test_causal_useful_flops_closed_forms():
    # dense causal: 4 * D * B * H * S(S+1)/2
    assert A.causal_useful_flops([(4096, 4096)] * 8, 256, 32) == 4 * 256 * 32 * 8 * 4096 * 4097 / 2
    # the long ring workload: 1.7593e13
    f = A.causal_useful_flops([(32768, 32768)], 128, 64)
    assert abs(f - 1.7593e13) / 1.7593e13 < 1e-4
    # non-causal: every pair
    assert A.causal_useful_flops([(3, 5)], 2, 1, causal=False) == 4 * 2 * 15
    # a shorter query block against more keys (top-left): sum min(i+1, S_kv)
    assert A.causal_useful_flops([(3, 2)], 1, 1) == 4 * (1 + 2 + 2)


# ---------------------------------------------------------------------- sliding window
def brute_window(q, k, v, scale, window):
    """Triple loop over (query, key, d): key j counts for query i iff i - window <= j <= i."""
    B, S, h_q, D = q.shape
    G = h_q // k.shape[2]
    O = np.zeros(q.shape[:3] + (v.shape[3],))
    L = np.zeros((B, h_q, S))
    for b in range(B):
        for h in range(h_q):
            g = h // G
            for i in range(S):
                scores = [(j, scale * sum(float(q[b, i, h, d]) * float(k[b, j, g, d]) for d in range(D)))
                          for j in range(S) if i - window <= j <= i]
                mx = max(sc for _, sc in scores)
                den = sum(math.exp(sc - mx) for _, sc in scores)
                for e in range(v.shape[3]):
                    O[b, i, h, e] = sum(math.exp(sc - mx) * float(v[b, j, g, e]) for j, sc in scores) / den
                L[b, h, i] = mx + math.log(den)
    return O, L


@pytest.mark.parametrize("window", [0, 1, 3, 11, 40])
def test_window_oracle_matches_brute_force(window):
    rng = np.random.default_rng(window + 5)
    q, k, v = rng.standard_normal((1, 12, 2, 4)), rng.standard_normal((1, 12, 1, 4)), rng.standard_normal((1, 12, 1, 5))
    O, L = A.attention(q, k, v, 0.7, causal=True, window=window)
    Ob, Lb = brute_window(q, k, v, 0.7, window)
    assert np.abs(O - Ob).max() < 1e-12 and np.abs(L - Lb).max() < 1e-12


@pytest.mark.parametrize("window", [0, 2, 7, 100])
def test_window_zero_queries_closed_form(window):
    """Q = 0: every visible key scores 0, so O_i is the mean of v over [i - window, i]
    and LSE_i = ln(min(i, window) + 1)."""
    rng = np.random.default_rng(9)
    S = 20
    q = np.zeros((2, S, 2, 8))
    k, v = rng.standard_normal((2, S, 1, 8)), rng.standard_normal((2, S, 1, 3))
    O, L = A.attention(q, k, v, 0.3, causal=True, window=window)
    for i in range(S):
        lo = max(0, i - window)
        assert np.abs(O[:, i, :, :] - v[:, lo:i + 1, 0, :].mean(axis=1)[:, None, :]).max() < 1e-12
        assert np.abs(L[:, :, i] - math.log(min(i, window) + 1)).max() < 1e-12


def test_window_zero_is_the_diagonal_and_large_window_is_causal():
    rng = np.random.default_rng(3)
    q, k, v = rng.standard_normal((1, 9, 1, 6)), rng.standard_normal((1, 9, 1, 6)), rng.standard_normal((1, 9, 1, 6))
    O0, L0 = A.attention(q, k, v, 0.5, causal=True, window=0)
    assert np.abs(O0 - v).max() < 1e-12  # each query sees only its own key
    assert np.abs(L0[0, 0] - 0.5 * np.einsum("sd,sd->s", q[0, :, 0], k[0, :, 0])).max() < 1e-12
    Ow, Lw = A.attention(q, k, v, 0.5, causal=True, window=8)
    Oc, Lc = A.attention(q, k, v, 0.5, causal=True)
    assert np.array_equal(Ow, Oc) and np.array_equal(Lw, Lc)


def test_window_useful_flops_closed_form():
    # w(w+1)/2 + (L - w)(w + 1) pairs when L > w
    L, w = 4096, 1000
    assert A.window_useful_flops(L, w, 128, 2) == 4.0 * 128 * 2 * (w * (w + 1) // 2 + (L - w) * (w + 1))
    assert A.window_useful_flops(50, 200, 64, 1) == A.causal_useful_flops([(50, 50)], 64, 1)
