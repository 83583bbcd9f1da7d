"""Planted mistakes: each plausible oracle bug must fail at least one pin (CPU only).

Every case swaps one helper of the oracle for a wrong variant (a dropped term,
a wrong sign or index, a transposed operand) and checks that the pin suite in
test_oracle_pins / test_oracle_schedule would catch it.  The mistakes are
planted in the oracle, on the CPU, and only for the duration of one test.
"""

import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import schedule as S
from tests.test_oracle_pins import brute_attention, brute_window

RNG = np.random.default_rng(7)


def _pins_pass():
    """A compact re-run of the value pins; True iff all of them hold."""
    try:
        for causal in (False, True):
            for h_q, h_kv in ((4, 2), (2, 2)):
                q = RNG.standard_normal((1, 9, h_q, 5))
                k = RNG.standard_normal((1, 9, h_kv, 5))
                v = RNG.standard_normal((1, 9, h_kv, 6))
                O, L = A.attention(q, k, v, 0.4, causal)
                Ob, Lb = brute_attention(q, k, v, 0.4, causal)
                if not (np.allclose(O, Ob, atol=1e-10) and np.allclose(L, Lb, atol=1e-10)):
                    return False
        q = RNG.standard_normal((1, 12, 2, 4))
        k = RNG.standard_normal((1, 12, 1, 4))
        v = RNG.standard_normal((1, 12, 1, 4))
        parts = [A.partial(q, k, v, 0.5, True, 0, lo, hi) for lo, hi in [(0, 4), (4, 9), (9, 12)]]
        O, L = A.merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]),
                       np.stack([p[2] for p in parts]))
        Ob, Lb = brute_attention(q, k, v, 0.5, True)
        if not (np.allclose(O, Ob, atol=1e-10) and np.allclose(L, Lb, atol=1e-10)):
            return False
        w = S.tile_walk(256, 384, 0, 512, 128, True, 4)
        if w != [(2, 256, 384), (0, 0, 128), (1, 128, 256)]:
            return False
        for window in (0, 3):
            q = RNG.standard_normal((1, 10, 2, 4))
            k = RNG.standard_normal((1, 10, 1, 4))
            v = RNG.standard_normal((1, 10, 1, 3))
            O, L = A.attention(q, k, v, 0.6, True, window=window)
            Ob, Lb = brute_window(q, k, v, 0.6, window)
            if not (np.allclose(O, Ob, atol=1e-10) and np.allclose(L, Lb, atol=1e-10)):
                return False
        # a sliding window of 100 keys: a Q tile at rows [512, 640) sees keys from 412 on
        if S.tile_walk(512, 640, 0, 1024, 128, True, 1, window=100) != [(0, 384, 512), (0, 512, 640)]:
            return False
        return True
    except Exception:
        return False


def test_unmutated_oracle_passes():
    assert _pins_pass()


def _scores_transposed(q_rows, k_rows, scale):
    # reads K's axes the wrong way round when it can: the "reshape, not transpose" mistake
    kk = k_rows.reshape(k_rows.shape[1], k_rows.shape[0]).T
    return scale * (q_rows @ kk.T)


MUTANTS = {
    # interleaved head groups (h mod h_kv) instead of contiguous ones; the pins use h_kv == G == 2
    "gqa_interleaved_groups": ("_kv_head", lambda h, g: h % g),
    "causal_strict": ("_visible", lambda qp, kp, c, w=None: (kp[None, :] < qp[:, None]) if c else np.ones((qp.size, kp.size), bool)),
    "causal_reversed": ("_visible", lambda qp, kp, c, w=None: (kp[None, :] >= qp[:, None]) if c else np.ones((qp.size, kp.size), bool)),
    # sliding window one key short (strict lower bound) and window ignored
    "window_strict": ("_visible", lambda qp, kp, c, w=None: (kp[None, :] <= qp[:, None]) & (
        (kp[None, :] > qp[:, None] - w) if w is not None else True) if c else np.ones((qp.size, kp.size), bool)),
    "window_ignored": ("_visible", lambda qp, kp, c, w=None: (kp[None, :] <= qp[:, None]) if c else np.ones((qp.size, kp.size), bool)),
    "scale_dropped": ("_scores", lambda q, k, s: q @ k.T),
    "scale_inverted": ("_scores", lambda q, k, s: (q @ k.T) / s),
    "k_reshaped_not_transposed": ("_scores", _scores_transposed),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_attention_mistakes_are_caught(monkeypatch, name):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(A, attr, fn)
    assert not _pins_pass(), name


def _merge_drops_step_factor(m, l, o, m_s, l_s, o_s):
    m_new = np.maximum(m, m_s)
    a = np.exp(m - m_new)
    return m_new, l * a + l_s, o * a[..., None] + o_s


def _merge_sign_flip(m, l, o, m_s, l_s, o_s):
    m_new = np.maximum(m, m_s)
    a = np.exp(m_new - m)
    b = np.exp(m_s - m_new)
    return m_new, l * a + l_s * b, o * a[..., None] + o_s * b[..., None]


def _merge_keeps_old_max(m, l, o, m_s, l_s, o_s):
    a = np.exp(m_s - np.maximum(m, m_s))
    return m, l + l_s * a, o + o_s * a[..., None]


@pytest.mark.parametrize("fn", [_merge_drops_step_factor, _merge_sign_flip, _merge_keeps_old_max])
def test_planted_merge_mistakes_are_caught(monkeypatch, fn):
    monkeypatch.setattr(A, "_merge_pair", fn)
    assert not _pins_pass()


def test_planted_schedule_mistakes_are_caught(monkeypatch):
    # ring starting at chunk 0 instead of the tile's own chunk
    monkeypatch.setattr(S, "ring_start_chunk", lambda *a, **k: 0)
    assert not _pins_pass()
    monkeypatch.undo()
    # visibility test that ignores causality
    monkeypatch.setattr(S, "pair_visible_in", lambda q_lo, q_hi, k_lo, k_hi, causal, *a: q_hi > q_lo and k_hi > k_lo)
    assert not _pins_pass()
    monkeypatch.undo()
    # window lower bound taken from the Q tile's last row instead of its first
    real = S.pair_visible_in

    def late_floor(q_lo, q_hi, k_lo, k_hi, causal, q_pos0=0, kv_pos0=0, window=None):
        if window is None:
            return real(q_lo, q_hi, k_lo, k_hi, causal, q_pos0, kv_pos0)
        return real(q_hi - 1, q_hi, k_lo, k_hi, causal, q_pos0, kv_pos0, window)
    monkeypatch.setattr(S, "pair_visible_in", late_floor)
    assert not _pins_pass()


def test_lse_missing_max_term_is_caught():
    """LSE = ln l alone (dropping m) differs from brute force whenever m != 0."""
    q = RNG.standard_normal((1, 5, 1, 3)) * 3
    k = RNG.standard_normal((1, 5, 1, 3))
    v = RNG.standard_normal((1, 5, 1, 3))
    m, l, _ = A.partial(q, k, v, 1.0, False)
    _, Lb = brute_attention(q, k, v, 1.0, False)
    assert not np.allclose(np.log(l), Lb, atol=1e-6)
    assert np.allclose(m + np.log(l), Lb, atol=1e-12)
    assert math.isfinite(float(m.max()))
