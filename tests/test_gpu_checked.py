"""The checked debug build, libattn_checked.so, on the GPU.

The checked variant compiles the same kernels with every global store index, TMA
tile coordinate and worklist index tested against its extent; a failed test
records ATTN_ERR_BOUNDS and skips the access (include/attn.h, "Checked builds").
These tests run the GPU parity suite and the full-size sampled tests against that
variant in a child process (ATTN_LIBRARY=checked), whose module fixtures assert a
clean device status, and show that the check reports and skips an out-of-range
store.
"""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def _checked_env():
    from ring_attention_online_gb300 import build as b
    if not os.path.exists(b.LIBS[True]):
        b.build(checked=True)
    env = dict(os.environ, ATTN_LIBRARY="checked")
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    return env


def _run(code_or_args, env, timeout=900):
    return subprocess.run([sys.executable, *code_or_args], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=timeout)


def test_checked_build_reports_and_skips_an_out_of_range_store():
    code = (
        "import torch, ring_attention_online_gb300 as ra\n"
        "assert ra.attn_build_checked()\n"
        "buf = torch.zeros(1, dtype=torch.int32, device='cuda')\n"
        "assert ra.attn_last_device_status() == 0\n"
        "ra.attn_selftest_bounds(buf)\n"
        "st = ra.attn_last_device_status()\n"
        "assert st == 6, st  # ATTN_ERR_BOUNDS, reported once\n"
        "assert ra.attn_last_device_status() == 0\n"
        "assert int(buf.item()) == 0  # the store was skipped\n"
        "print('ok')\n")
    r = _run(["-c", code], _checked_env(), timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr


def test_parity_suites_run_clean_on_the_checked_build():
    """Every GPU parity case and every full-size sampled case, element by element against
    the oracle as in the ordinary suite, with every index checked: the suites' module
    fixtures assert that the device status is clean at the end."""
    r = _run(["-m", "pytest", "tests/test_gpu_parity.py", "tests/test_gpu_fullsize.py", "-m", "gpu", "-x", "-q",
              "-p", "no:cacheprovider"], _checked_env())
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and "failed" not in r.stdout, tail
