"""attn_decode_splitkv_noalloc: split-KV decode for callers that cannot allocate.

Some callers cannot hand the library device memory: their host framework owns all
device memory, or they run latency-critical loops that must not call cudaMalloc or
cudaFree (both can synchronise the device).  This entry point keeps the decode
partials in a fixed array of device memory inside the library instead of a
workspace argument.  The test calls it twice in a row through the C ABI (so the
second call runs on whatever the first left in the shared array) and checks each
result against attn_decode_splitkv with a caller workspace, within the parity
tolerance of the other GPU tests.  It lives in a file collected last and passes
both alone in a fresh process and after the rest of the suite.
"""

import ctypes

import numpy as np
import pytest
import torch

import ring_attention_online_gb300 as ra
import synthetic as syn

pytestmark = pytest.mark.gpu

TOL_MAX, TOL_MEAN, TOL_LSE = 1e-2, 1e-3, 1e-3


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_noalloc_decode_matches_workspace_decode_on_two_calls():
    lib = ra.load_library()
    cases = [  # (B, S_kv, h_q, h_kv, D, num_splits, seed)
        (2, 5000, 16, 2, 128, 7, 101),
        (3, 2500, 8, 1, 64, 16, 202),
    ]
    for B, S_kv, h_q, h_kv, D, splits, seed in cases:
        q, k, v = syn.qkv((B, h_q, D), (B, S_kv, h_kv, D), "bf16", seed, "cuda")
        scale = float(D) ** -0.5
        o_ref = torch.empty_like(q)
        lse_ref = torch.empty(B, h_q, device="cuda")
        ws = torch.empty(ra.attn_decode_workspace_bytes(B, h_q, D, splits), dtype=torch.uint8, device="cuda")
        st = lib.attn_decode_splitkv(_p(q), _p(k), _p(v), _p(o_ref), _p(lse_ref), B, S_kv, h_q, h_kv, D, 1, scale,
                                     splits, _p(ws), ws.numel(), _stream())
        assert st == 0
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, h_q), float("nan"), device="cuda")
        st = lib.attn_decode_splitkv_noalloc(_p(q), _p(k), _p(v), _p(o), _p(lse), B, S_kv, h_q, h_kv, D, 1, scale,
                                             splits, _stream())
        assert st == 0
        torch.cuda.synchronize()
        got, ref = o.float().cpu().numpy(), o_ref.float().cpu().numpy()
        assert np.isfinite(got).all()
        err = np.abs(got - ref)
        assert err.max() <= TOL_MAX and err.mean() <= TOL_MEAN
        assert np.abs(lse.cpu().numpy() - lse_ref.cpu().numpy()).max() <= TOL_LSE
    assert ra.attn_last_device_status() == 0


def test_noalloc_decode_rejects_partials_larger_than_its_scratch():
    lib = ra.load_library()
    need = ra.attn_decode_workspace_bytes(8, 64, 128, 64)  # about 17 MB of partials
    assert need > 16 * 1024 * 1024
    q = torch.zeros(8, 64, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(8, 64, 8, 128, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    st = lib.attn_decode_splitkv_noalloc(_p(q), _p(k), _p(k), _p(o), None, 8, 64, 64, 8, 128, 1, 0.1, 64, _stream())
    assert st == 2  # ATTN_ERR_UNSUPPORTED, nothing launched
