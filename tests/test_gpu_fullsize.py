"""GPU parity at the workloads' full sizes, in the launch configuration bench.py times.

Each workload runs exactly as bench.py runs it (same synthetic inputs, seed 0, same
entry point and arguments); the fp64 oracle then recomputes sampled outputs one by
one: chosen rows of chosen (batch, head) pairs against all of their keys, whole
sampled sequences (jagged), and sampled (batch, query head) rows of the decode.
Samples include the first and last rows, rows on both sides of 128-row tile edges and
of ring-chunk edges, and random ones.  Same tolerances as the small-size parity tests.
"""

import math

import numpy as np
import pytest
import torch

import ring_attention_online_gb300 as ra
import synthetic as syn
from oracle import attention as A

pytestmark = pytest.mark.gpu

TOL_MAX, TOL_MEAN, TOL_LSE = 1e-2, 1e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ra.load_library()
    yield
    assert ra.attn_last_device_status() == 0


def _rows(S, rng, extra=()):
    edges = [0, 1, 127, 128, 129, 255, 256, S // 2, S - 129, S - 128, S - 2, S - 1, *extra]
    rnd = rng.integers(0, S, 8)
    return np.unique(np.clip(np.concatenate([edges, rnd]), 0, S - 1))


def _check(o_got, lse_got, O, L, what):
    err = np.abs(o_got.astype(np.float64) - O)
    assert np.isfinite(o_got).all(), what
    assert err.max() <= TOL_MAX, f"{what}: max err {err.max():.3e}"
    assert err.mean() <= TOL_MEAN, f"{what}: mean err {err.mean():.3e}"
    assert np.abs(lse_got.astype(np.float64) - L).max() <= TOL_LSE, what


def _prefill_sampled(name, samples, extra_rows=(), window=None):
    cfg = syn.WORKLOADS[name]
    q, k, v = syn.prefill_inputs(cfg, seed=0, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(cfg["B"], cfg["h_q"], cfg["S_q"], device="cuda", dtype=torch.float32)
    if window is None:
        ra.attn_prefill(q, k, v, o, lse, causal=cfg["causal"], num_chunks=cfg["num_chunks"])
    else:
        ra.attn_prefill_window(q, k, v, o, lse, window=window, num_chunks=cfg["num_chunks"])
    torch.cuda.synchronize()
    assert ra.attn_last_device_status() == 0
    G = cfg["h_q"] // cfg["h_kv"]
    scale = 1 / math.sqrt(cfg["D"])
    rng = np.random.default_rng(11)
    for b, h in samples:
        g = h // G
        rows = _rows(cfg["S_q"], rng, extra_rows)
        qc = q[b:b + 1, :, h:h + 1].cpu()
        kc, vc = k[b:b + 1, :, g:g + 1].cpu(), v[b:b + 1, :, g:g + 1].cpu()
        O, L = A.attention(qc, kc, vc, scale, cfg["causal"], rows=rows, window=window)
        _check(o[b, rows, h].float().cpu().numpy(), lse[b, h, rows].cpu().numpy(), O[0, rows, 0], L[0, 0, rows],
               f"{name} b={b} h={h}")
    del q, k, v, o, lse
    torch.cuda.empty_cache()


def test_dense_causal_b8_h32_s4096_d256_sampled():
    _prefill_sampled("dense_causal_b8_h32_s4096_d256", [(0, 0), (3, 17), (7, 31)])


def test_long_gqa_ring8_s32768_sampled():
    # rows at the 4096-key ring-chunk edges too; heads of two different KV groups
    chunk_edges = [c * 4096 + d for c in range(1, 8) for d in (-1, 0)]
    _prefill_sampled("long_gqa_ring8_s32768_hq64_hkv8_d128", [(0, 0), (0, 1), (0, 37), (0, 63)], chunk_edges)


def test_window4096_gqa_s32768_sampled():
    cfg = syn.WORKLOADS["window4096_gqa_s32768_hq64_hkv8_d128"]
    w = cfg["window"]
    _prefill_sampled("window4096_gqa_s32768_hq64_hkv8_d128", [(0, 2), (0, 45)], (w - 1, w, w + 1, w + 128),
                     window=w)


def test_jagged_1152seq_sampled_sequences():
    cfg = syn.WORKLOADS["jagged_causal_1152seq_h4_d128"]
    q, k, v, offs = syn.jagged_inputs(cfg, seed=0, device="cuda")
    T = int(offs[-1])
    lens = np.diff(offs.astype(np.int64))
    o = torch.empty_like(q)
    lse = torch.empty(cfg["H"], T, device="cuda", dtype=torch.float32)
    offs_d = torch.from_numpy(offs).to("cuda")
    ws = torch.empty(ra.attn_jagged_workspace_bytes(len(lens), T, int(lens.max())), dtype=torch.uint8, device="cuda")
    ra.attn_jagged(q, k, v, o, offs_d, int(lens.max()), ws, lse, causal=True)
    torch.cuda.synchronize()
    assert ra.attn_last_device_status() == 0
    rng = np.random.default_rng(12)
    seqs = sorted({int(np.argmax(lens)), int(np.argmin(lens)), 0, len(lens) - 1, *rng.integers(0, len(lens), 6)})
    scale = 1 / math.sqrt(cfg["D"])
    for sq in seqs:
        lo, hi = int(offs[sq]), int(offs[sq + 1])
        O, L = A.attention(q[None, lo:hi].cpu(), k[None, lo:hi].cpu(), v[None, lo:hi].cpu(), scale, True)
        _check(o[lo:hi].float().cpu().numpy(), lse[:, lo:hi].cpu().numpy(), O[0], L[0], f"jagged seq {sq}")


def test_decode_b8_kv1m_sampled():
    cfg = syn.WORKLOADS["decode_splitkv_b8_hq64_hkv8_d128_kv1m"]
    q, k, v = syn.decode_inputs(cfg, seed=0, device="cuda")
    B, h_q, h_kv, D, C = cfg["B"], cfg["h_q"], cfg["h_kv"], cfg["D"], cfg["num_splits"]
    o = torch.empty_like(q)
    lse = torch.empty(B, h_q, device="cuda", dtype=torch.float32)
    ws = torch.empty(ra.attn_decode_workspace_bytes(B, h_q, D, C), dtype=torch.uint8, device="cuda")
    ra.attn_decode_splitkv(q, k, v, o, ws, lse, num_splits=C)
    torch.cuda.synchronize()
    assert ra.attn_last_device_status() == 0
    G = h_q // h_kv
    scale = 1 / math.sqrt(D)
    for b, h in [(0, 0), (5, 42), (7, 63)]:
        g = h // G
        # the 8 query heads of the KV group against all 1 048 576 keys, in the page's
        # split-and-merge form (exact up to rounding)
        O, L = A.decode(q[b:b + 1, g * G:(g + 1) * G].cpu(), k[b:b + 1, :, g:g + 1].cpu(),
                        v[b:b + 1, :, g:g + 1].cpu(), scale, C)
        _check(o[b:b + 1, g * G:(g + 1) * G].float().cpu().numpy(), lse[b:b + 1, g * G:(g + 1) * G].cpu().numpy(),
               O, L, f"decode b={b} group={g}")
    del q, k, v
    torch.cuda.empty_cache()
