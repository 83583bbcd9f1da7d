"""Blockwise online-softmax attention on one GB300 (sm_103a).

The computation runs in `libattn.so` (hand-written CUDA kernels: tcgen05/TMEM/TMA
prefill, split-KV decode, triplet merge, jagged worklist builder).  This module
only marshals arguments to its C ABI (include/attn.h): each function below has
the name of the C entry point it calls, takes torch tensors that already live on
the GPU, and raises AttnError on a non-OK status.  Nothing here computes
attention, and there is no fallback: if the library is not built, loading it
raises.

Layouts (contiguous): Q/O [B, S_q, h_q, D]; K/V [B, S_kv, h_kv, D];
LSE, m, l [B, h_q, S_q] fp32; jagged Q/K/V/O [T, H, D], jagged LSE [H, T].
"""

from __future__ import annotations

import ctypes
import math
import os

__all__ = [
    "AttnError", "load_library", "library_path",
    "attn_prefill", "attn_prefill_window", "attn_partial", "attn_merge", "attn_jagged", "attn_decode_splitkv",
    "attn_jagged_workspace_bytes", "attn_decode_workspace_bytes", "attn_decode_splitkv_noalloc",
    "attn_last_device_status", "attn_status_string", "attn_tile_walk", "attn_selftest_wait_timeout",
    "attn_probe_mma_cycles", "attn_build_checked", "attn_selftest_bounds",
    "BLOCK_M", "BLOCK_N", "STATUS",
]

BLOCK_M = 128
BLOCK_N = 128
STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_CUDA",
          4: "ATTN_ERR_TIMEOUT", 5: "ATTN_ERR_DEVICE_INPUT", 6: "ATTN_ERR_BOUNDS"}
_FP16, _BF16 = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


def library_path() -> str:
    """libattn.so, or its checked debug variant libattn_checked.so when the
    environment variable ATTN_LIBRARY is "checked" (see attn.h, "Checked builds")."""
    variant = os.environ.get("ATTN_LIBRARY", "")
    if variant not in ("", "default", "checked"):
        raise ValueError(f"ATTN_LIBRARY={variant!r}: expected 'checked' or unset")
    return os.path.join(_HERE, "libattn_checked.so" if variant == "checked" else "libattn.so")


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


_P, _I, _F, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_SIGNATURES = {
    "attn_prefill": [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P],
    "attn_partial": [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _I, _P],
    "attn_merge": [_P, _P, _P, _I, _I, _I, _I, _I, _P, _I, _P, _P],
    "attn_jagged": [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _S, _P],
    "attn_jagged_workspace_bytes": [_I, _I, _I],
    "attn_decode_splitkv": [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _S, _P],
    "attn_decode_workspace_bytes": [_I, _I, _I, _I],
    "attn_decode_splitkv_noalloc": [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P],
    "attn_last_device_status": [_P],
    "attn_status_string": [_I],
    "attn_prefill_window": [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P],
    "attn_tile_walk": [_I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _I, _P],
    "attn_selftest_wait_timeout": [ctypes.c_uint64, _P],
    "attn_probe_mma_cycles": [_P, _I, _P],
    "attn_build_checked": [],
    "attn_selftest_bounds": [_P, _P],
}


def load_library():
    """Load libattn.so (once).  Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it with `python -m ring_attention_online_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, args in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_size_t if name.endswith("_bytes") else (
                ctypes.c_char_p if name == "attn_status_string" else ctypes.c_int)
        _LIB = lib
    return _LIB


# ------------------------------------------------------------------ marshalling
def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return _FP16
    if t.dtype == torch.bfloat16:
        return _BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream, t):
    import torch
    s = torch.cuda.current_stream(t.device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _check(status: int, where: str):
    if status != 0:
        raise AttnError(status, where)


def _cuda_contig(*ts):
    for t in ts:
        if t is not None:
            _need(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")


def _scale(scale, D):
    return 1.0 / math.sqrt(D) if scale is None else float(scale)


# ------------------------------------------------------------------ entry points
def attn_prefill(q, k, v, o, lse=None, *, scale=None, causal=False, num_chunks=1, stream=None):
    """Prefill attention with a ring-order walk over num_chunks KV chunks (see attn.h)."""
    _cuda_contig(q, k, v, o, lse)
    B, S_q, h_q, D = q.shape
    S_kv, h_kv = k.shape[1], k.shape[2]
    _need(k.shape == v.shape and o.shape == q.shape and k.shape[0] == B and k.shape[3] == D, "shape mismatch")
    st = load_library().attn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, S_q, S_kv, h_q, h_kv, D,
                                     _dtype_code(q), _scale(scale, D), int(bool(causal)), int(num_chunks),
                                     _stream(stream, q))
    _check(st, "attn_prefill")


def attn_prefill_window(q, k, v, o, lse=None, *, window, scale=None, num_chunks=1, stream=None):
    """Causal prefill where query i sees keys i - window .. i (see attn.h)."""
    _cuda_contig(q, k, v, o, lse)
    B, S_q, h_q, D = q.shape
    S_kv, h_kv = k.shape[1], k.shape[2]
    _need(k.shape == v.shape and o.shape == q.shape and k.shape[0] == B and k.shape[3] == D, "shape mismatch")
    st = load_library().attn_prefill_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, S_q, S_kv, h_q, h_kv,
                                            D, _dtype_code(q), _scale(scale, D), int(window), int(num_chunks),
                                            _stream(stream, q))
    _check(st, "attn_prefill_window")


def attn_partial(q, k, v, m, l, o_unnorm, *, scale=None, causal=False, q_pos0=0, kv_begin=0, kv_end=None,
                 stream=None):
    """Partial triplet (m, l, unnormalised O) of keys [kv_begin, kv_end) (see attn.h)."""
    _cuda_contig(q, k, v, m, l, o_unnorm)
    B, S_q, h_q, D = q.shape
    S_kv, h_kv = k.shape[1], k.shape[2]
    kv_end = S_kv if kv_end is None else kv_end
    st = load_library().attn_partial(_ptr(q), _ptr(k), _ptr(v), _ptr(m), _ptr(l), _ptr(o_unnorm), B, S_q, S_kv,
                                     h_q, h_kv, D, _dtype_code(q), _scale(scale, D), int(bool(causal)),
                                     int(q_pos0), int(kv_begin), int(kv_end), _stream(stream, q))
    _check(st, "attn_partial")


def attn_merge(m, l, o_unnorm, out, lse=None, *, stream=None):
    """Fold stacked partials m,l [C,B,H,S_q], o [C,B,S_q,H,D] into out [B,S_q,H,D] (see attn.h)."""
    _cuda_contig(m, l, o_unnorm, out, lse)
    C, B, S_q, H, D = o_unnorm.shape
    _need(tuple(m.shape) == (C, B, H, S_q) and tuple(l.shape) == (C, B, H, S_q), "m/l shape mismatch")
    st = load_library().attn_merge(_ptr(m), _ptr(l), _ptr(o_unnorm), C, B, S_q, H, D, _ptr(out), _dtype_code(out),
                                   _ptr(lse), _stream(stream, out))
    _check(st, "attn_merge")


def attn_jagged_workspace_bytes(num_seqs: int, total_tokens: int, max_seqlen: int) -> int:
    return int(load_library().attn_jagged_workspace_bytes(num_seqs, total_tokens, max_seqlen))


def attn_jagged(q, k, v, o, seq_offsets, max_seqlen, workspace, lse=None, *, scale=None, causal=True,
                stream=None):
    """Jagged self-attention over packed sequences (see attn.h)."""
    _cuda_contig(q, k, v, o, lse, seq_offsets, workspace)
    T, H, D = q.shape
    num_seqs = seq_offsets.numel() - 1
    st = load_library().attn_jagged(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(seq_offsets), num_seqs, T,
                                    int(max_seqlen), H, D, _dtype_code(q), _scale(scale, D), int(bool(causal)),
                                    _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream, q))
    _check(st, "attn_jagged")


def attn_decode_workspace_bytes(B: int, h_q: int, D: int, num_splits: int) -> int:
    return int(load_library().attn_decode_workspace_bytes(B, h_q, D, num_splits))


def attn_decode_splitkv(q, k, v, o, workspace, lse=None, *, num_splits, scale=None, stream=None):
    """Split-KV decode: q [B,h_q,D] against k/v [B,S_kv,h_kv,D] (see attn.h)."""
    _cuda_contig(q, k, v, o, lse, workspace)
    B, h_q, D = q.shape
    S_kv, h_kv = k.shape[1], k.shape[2]
    st = load_library().attn_decode_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, S_kv, h_q, h_kv, D,
                                            _dtype_code(q), _scale(scale, D), int(num_splits), _ptr(workspace),
                                            workspace.numel() * workspace.element_size(), _stream(stream, q))
    _check(st, "attn_decode_splitkv")


def attn_decode_splitkv_noalloc(q, k, v, o, lse=None, *, num_splits, scale=None, stream=None):
    """attn_decode_splitkv with the partials in the library's fixed device scratch, for
    callers that cannot allocate device memory (see attn.h for its limit and sharing rules)."""
    _cuda_contig(q, k, v, o, lse)
    B, h_q, D = q.shape
    S_kv, h_kv = k.shape[1], k.shape[2]
    st = load_library().attn_decode_splitkv_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, S_kv, h_q,
                                                    h_kv, D, _dtype_code(q), _scale(scale, D), int(num_splits),
                                                    _stream(stream, q))
    _check(st, "attn_decode_splitkv_noalloc")


def attn_last_device_status(stream=None) -> int:
    """Synchronise, then return (and clear) the device-side status code."""
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(load_library().attn_last_device_status(ctypes.c_void_p(s.cuda_stream)))


def attn_selftest_wait_timeout(timeout_ns: int, stream=None):
    """Run the bounded-wait self-test kernel (see attn.h); read the result with attn_last_device_status()."""
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    _check(load_library().attn_selftest_wait_timeout(int(timeout_ns), ctypes.c_void_p(s.cuda_stream)),
           "attn_selftest_wait_timeout")


def attn_probe_mma_cycles(groups: int = 4096, stream=None) -> float:
    """Cycles per tcgen05 kind::f16 M=128 N=128 K=16 MMA issued back to back on one SM
    (see attn.h); the per-SM dense bf16 rate is 128*128*16*2 / this."""
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    out = torch.zeros(2, dtype=torch.int64, device=s.device)
    _check(load_library().attn_probe_mma_cycles(ctypes.c_void_p(out.data_ptr()), int(groups),
                                                ctypes.c_void_p(s.cuda_stream)), "attn_probe_mma_cycles")
    s.synchronize()
    cycles, gave_up = (int(x) for x in out.cpu().tolist())
    if gave_up:
        raise AttnError(4, "attn_probe_mma_cycles")
    return cycles / (8.0 * int(groups))


def attn_build_checked() -> bool:
    """True when the loaded library is the checked debug variant."""
    return bool(load_library().attn_build_checked())


def attn_selftest_bounds(buf, stream=None):
    """Checked variant only: a store to index 1 of the one-element int32 CUDA tensor
    `buf` through the store check (see attn.h); read the result with
    attn_last_device_status()."""
    import torch
    _need(buf.is_cuda and buf.dtype == torch.int32 and buf.numel() == 1, "buf: one int32 CUDA element")
    s = torch.cuda.current_stream() if stream is None else stream
    _check(load_library().attn_selftest_bounds(_ptr(buf), ctypes.c_void_p(s.cuda_stream)), "attn_selftest_bounds")


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def attn_tile_walk(q_lo, q_hi, kv_lo, kv_hi, *, block_n=BLOCK_N, causal=True, num_chunks=1, q_pos0=0, kv_pos0=0,
                   window=None):
    """KV tiles (chunk, tile_start, mask_end) one Q tile visits, from the library's scheduler (host code)."""
    lib = load_library()
    n = ctypes.c_int(0)
    w = -1 if window is None else int(window)
    st = lib.attn_tile_walk(q_lo, q_hi, kv_lo, kv_hi, block_n, int(bool(causal)), num_chunks, q_pos0, kv_pos0, w,
                            None, None, None, 0, ctypes.byref(n))
    _check(st, "attn_tile_walk")
    cap = n.value
    arr = [(ctypes.c_int * max(cap, 1))() for _ in range(3)]
    st = lib.attn_tile_walk(q_lo, q_hi, kv_lo, kv_hi, block_n, int(bool(causal)), num_chunks, q_pos0, kv_pos0, w,
                            arr[0], arr[1], arr[2], cap, ctypes.byref(n))
    _check(st, "attn_tile_walk")
    return [(arr[0][i], arr[1][i], arr[2][i]) for i in range(cap)]
