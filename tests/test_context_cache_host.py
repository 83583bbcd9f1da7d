"""Host-only check of the per-context address cache behind attn_decode_splitkv_noalloc.

The no-allocation decode keeps the device address of its scratch array per device,
recorded under the id of the CUDA context it was looked up in.  After a device reset
the next context has a new id (its handle value may be reused, its id is not), and the
cached address must not be handed out for it.  This compiles the header with g++ and
checks that contract with made-up ids and addresses: no GPU, no CUDA call.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "ring_attention_online_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "context_cache.h"

static int fails = 0;
#define CHECK(c) do { if (!(c)) { std::printf("FAIL line %d: %s\n", __LINE__, #c); ++fails; } } while (0)

int main() {
  attn::ContextAddressCache<4> c;
  int a = 0, b = 0;
  void* pa = &a;
  void* pb = &b;
  CHECK(c.get(0, 7) == nullptr);               // nothing recorded yet
  CHECK(c.put(0, 7, pa));
  CHECK(c.get(0, 7) == pa);                    // same device, same context
  CHECK(c.get(0, 8) == nullptr);               // a new context after a reset: stale
  CHECK(c.get(1, 7) == nullptr);               // another device
  CHECK(c.put(0, 8, pb));                      // the fresh lookup replaces the entry
  CHECK(c.get(0, 8) == pb);
  CHECK(c.get(0, 7) == nullptr);               // the old context's entry is gone
  CHECK(c.put(3, 0, pa) && c.get(3, 0) == pa); // id 0 is an ordinary id
  CHECK(c.get(2, 0) == nullptr);               // untouched device with id 0
  CHECK(!c.put(4, 1, pa) && c.get(4, 1) == nullptr);   // out of range
  CHECK(!c.put(-1, 1, pa) && c.get(-1, 1) == nullptr);
  CHECK(!c.put(1, 1, nullptr) && c.get(1, 1) == nullptr);  // null is never recorded
  std::printf(fails ? "FAILED\n" : "OK\n");
  return fails ? 1 : 0;
}
"""


def test_context_cache_never_returns_an_address_of_another_context(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    src = tmp_path / "cache_test.cc"
    exe = tmp_path / "cache_test"
    src.write_text(PROGRAM)
    r = subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-I", HEADER_DIR, str(src), "-o", str(exe), "-pthread"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout
