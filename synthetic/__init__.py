"""Seeded synthetic inputs for the tests, the bench and the smoke check.

This module only draws numbers and sequence lengths; it holds none of the
attention arithmetic, so both the CUDA path's tests and the fp64 oracle can
take their inputs from it without sharing any computation.

Recipe (the pages publish no data; every input is synthetic):
  * Q, K, V ~ N(0, 1), drawn in fp32 with a torch.Generator seeded with `seed`
    on the target device, in the order q, k, v, then cast to fp16 or bf16.
    Large tensors are drawn slice by slice along their first axis with the
    same generator, so the stream stays deterministic for a given seed.
  * Jagged lengths ~ uniform integers in [lo, hi] from
    numpy.random.default_rng(seed), packed by an exclusive cumulative sum into
    int32 seq_offsets of length n + 1.
"""

from __future__ import annotations

import math

import numpy as np
import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}

# The pages' workloads, named by what they are.  Sizes follow the dense causal
# and jagged result tables of the Helion dependent-bounds page, the ring-KV
# GQA prefill page and the Llama-70B-style decode study of the mesh decode page.
WORKLOADS = {
    "tiny_gqa_ring4": dict(kind="prefill", B=1, S_q=256, S_kv=256, h_q=2, h_kv=1, D=64,
                           dtype="fp16", causal=False, num_chunks=4),
    "dense_causal_b8_h32_s4096_d256": dict(kind="prefill", B=8, S_q=4096, S_kv=4096, h_q=32,
                                           h_kv=32, D=256, dtype="bf16", causal=True,
                                           num_chunks=1),
    "jagged_causal_1152seq_h4_d128": dict(kind="jagged", num_seqs=1152, len_lo=64,
                                          len_hi=1024, H=4, D=128, dtype="bf16", causal=True),
    "long_gqa_ring8_s32768_hq64_hkv8_d128": dict(kind="prefill", B=1, S_q=32768, S_kv=32768,
                                                 h_q=64, h_kv=8, D=128, dtype="bf16",
                                                 causal=True, num_chunks=8),
    "decode_splitkv_b8_hq64_hkv8_d128_kv1m": dict(kind="decode", B=8, h_q=64, h_kv=8, D=128,
                                                  S_kv=1 << 20, dtype="bf16", num_splits=64),
    # the long GQA prefill with a causal sliding window of 4096 keys (no page states a
    # window workload; this is the long-context shape with a typical window size)
    "window4096_gqa_s32768_hq64_hkv8_d128": dict(kind="prefill", B=1, S_q=32768, S_kv=32768,
                                                 h_q=64, h_kv=8, D=128, dtype="bf16",
                                                 causal=True, num_chunks=1, window=4096),
}


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


def normal(shape, dtype, gen: torch.Generator, device) -> torch.Tensor:
    """N(0,1) drawn in fp32 slice by slice along axis 0, stored in `dtype`."""
    out = torch.empty(shape, dtype=dtype, device=device)
    rows = shape[0]
    per_row = max(1, math.prod(shape[1:]))
    step = max(1, (1 << 28) // per_row)  # at most ~1 GiB of fp32 per draw
    for lo in range(0, rows, step):
        hi = min(rows, lo + step)
        out[lo:hi] = torch.randn((hi - lo,) + tuple(shape[1:]), generator=gen,
                                 device=device, dtype=torch.float32).to(dtype)
    return out


def qkv(q_shape, kv_shape, dtype: str, seed: int = 0, device="cpu", v_shape=None):
    """q, k, v drawn in that order from one generator seeded with `seed`."""
    dt = DTYPES[dtype]
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q = normal(q_shape, dt, gen, device)
    k = normal(kv_shape, dt, gen, device)
    v = normal(v_shape or kv_shape, dt, gen, device)
    return q, k, v


def jagged_lengths(n: int, lo: int, hi: int, seed: int = 0) -> np.ndarray:
    """n lengths uniform in [lo, hi] (inclusive)."""
    return np.random.default_rng(seed).integers(lo, hi + 1, n).astype(np.int64)


def offsets_from_lengths(lengths) -> np.ndarray:
    """Exclusive cumulative sum, int32, length n + 1."""
    lengths = np.asarray(lengths, dtype=np.int64)
    offs = np.zeros(lengths.size + 1, dtype=np.int64)
    np.cumsum(lengths, out=offs[1:])
    return offs.astype(np.int32)


def prefill_inputs(cfg: dict, seed: int = 0, device="cpu"):
    """q [B,S_q,h_q,D], k, v [B,S_kv,h_kv,D] for a prefill workload."""
    return qkv((cfg["B"], cfg["S_q"], cfg["h_q"], cfg["D"]),
               (cfg["B"], cfg["S_kv"], cfg["h_kv"], cfg["D"]), cfg["dtype"], seed, device)


def jagged_inputs(cfg: dict, seed: int = 0, device="cpu"):
    """(q, k, v [T,H,D], seq_offsets int32 [n+1]) for a jagged workload."""
    offs = offsets_from_lengths(jagged_lengths(cfg["num_seqs"], cfg["len_lo"], cfg["len_hi"], seed))
    total = int(offs[-1])
    shape = (total, cfg["H"], cfg["D"])
    q, k, v = qkv(shape, shape, cfg["dtype"], seed, device)
    return q, k, v, offs


def decode_inputs(cfg: dict, seed: int = 0, device="cpu"):
    """q [B,h_q,D], k, v [B,S_kv,h_kv,D] for a decode workload."""
    return qkv((cfg["B"], cfg["h_q"], cfg["D"]),
               (cfg["B"], cfg["S_kv"], cfg["h_kv"], cfg["D"]), cfg["dtype"], seed, device)
