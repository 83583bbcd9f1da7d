"""Build libattn.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each .cu translation unit is compiled in parallel to _build/*.o, then linked
into ring_attention_online_gb300/libattn.so with the CUDA runtime linked
statically.  Re-running only recompiles units whose sources or headers changed.

The checked variant (build(checked=True), or --checked) compiles the same
sources with ATTN_CHECKED=1 into _build_checked/ and links
libattn_checked.so: its kernels test every global store index, TMA tile
coordinate and worklist index against its extent and report a violation as
ATTN_ERR_BOUNDS instead of making the access.  The Python binding loads it when
the environment variable ATTN_LIBRARY is "checked".

    python -m ring_attention_online_gb300.build [-v] [--checked | --all]
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBS = {False: os.path.join(PKG, "libattn.so"), True: os.path.join(PKG, "libattn_checked.so")}
BUILDS = {False: os.path.join(ROOT, "_build"), True: os.path.join(ROOT, "_build_checked")}

SOURCES = ["api.cu", "prefill_d64.cu", "prefill_d128.cu", "prefill_d256.cu", "merge.cu", "worklist.cu", "decode.cu",
           "decode_noalloc.cu", "probe.cu"]
HEADERS = ["common.cuh", "ptx.cuh", "schedule.cuh", "prefill_common.cuh", "prefill_pair_kernel.cuh", "merge.cuh",
           "context_cache.h", "prefill_cta2_kernel.cuh", "checked.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        raise RuntimeError("nvcc not found")
    return nvcc


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [src] + [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "attn.h"), __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, verbose: bool, checked: bool) -> str:
    obj = os.path.join(BUILDS[checked], os.path.splitext(src)[0] + ".o")
    path = os.path.join(CSRC, src)
    if _stale(obj, path):
        cmd = [_nvcc(), *ARCH, *FLAGS, *(["-DATTN_CHECKED=1"] if checked else []), "-c", path, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr, flush=True)
    return obj


def _link(objs, checked: bool) -> str:
    lib = LIBS[checked]
    if not os.path.exists(lib) or any(os.path.getmtime(o) > os.path.getmtime(lib) for o in objs):
        tmp = lib + ".tmp"
        cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


def build(verbose: bool = False, jobs: int | None = None, checked: bool = False, both: bool = False) -> str:
    """Compile every CUDA unit for sm_103a and link libattn.so (checked: libattn_checked.so;
    both: the two, compiled in one parallel pass); returns the path of the library built last."""
    variants = [False, True] if both else [checked]
    for v in variants:
        os.makedirs(BUILDS[v], exist_ok=True)
    work = [(src, v) for v in variants for src in SOURCES]
    jobs = jobs or min(len(work), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(jobs) as ex:
        objs = list(ex.map(lambda sv: _compile(sv[0], verbose, sv[1]), work))
    lib = None
    for v in variants:
        lib = _link([o for o, (_, vv) in zip(objs, work) if vv == v], v)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, checked="--checked" in sys.argv, both="--all" in sys.argv))
