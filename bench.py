#!/usr/bin/env python
"""Throughput of the blockwise online-softmax attention path on GB300.

Headline (one JSON line on rank 0): dense causal prefill B=8, H=32, S=4096,
D=256, bf16, 128x128 tiles with fully masked tiles pruned, in causal-useful
TFLOP/s (4 * D * B * H * S(S+1)/2 FLOPs per step).  The same line carries, under
"secondary", the other workloads of the pages at their full sizes: jagged causal
self-attention (1152 sequences), long GQA prefill with an 8-chunk ring-order
walk (S=32768), and split-KV decode (B=8, 1M keys, 64 splits, in HBM GB/s).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-secondary]

N > 1 runs under torch.distributed.run, one rank per GPU: every rank runs its own
copy of the workload (independent problems; no collective on the data path),
the timed region is bracketed by barriers and the max time over ranks is used.
--impl reference times the fp64 CPU oracle on the host cores on bounded samples
of the same workload.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal-useful TFLOP/s (prefill) and HBM GB/s (decode) on 1 GB300 vs roofline"
HEADLINE = "dense_causal_b8_h32_s4096_d256"
# measured after the headline in the same run, each with its own roofline
SECONDARY = ("jagged_causal_1152seq_h4_d128", "long_gqa_ring8_s32768_hq64_hkv8_d128",
             "decode_splitkv_b8_hq64_hkv8_d128_kv1m", "window4096_gqa_s32768_hq64_hkv8_d128")
# the pages' best pruned dense causal figure for this exact workload (Pallas backend,
# hardware not stated): context, not a target
PAGES_DENSE_CAUSAL_TFS = 225.8
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ plumbing
def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=HEADLINE, help="workload to report as the line (default: headline)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the batch / sequence count (smaller cases for profiling)")
    ap.add_argument("--seq", type=int, default=None,
                    help="override a prefill workload's sequence length (smaller cases for profiling)")
    return ap.parse_args(argv)


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank scalar over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_units: float, per_rank_ms: float, world: int, device=None):
    """Whole-job throughput: units all ranks processed / max time over ranks."""
    ms = max_over_ranks(per_rank_ms, device)
    return per_rank_units * world, ms


# Nominal denominators, beside the measured ones: dense bf16 tcgen05 rate per SM
# (a 128x128x16 kind::f16 MMA issues every 64 cycles back to back on one SM, as a
# microbenchmark on this GPU confirmed) x SMs x the maximum SM clock, and the
# published HBM3e bandwidth.
BF16_FLOP_PER_CLK_PER_SM = 128 * 128 * 16 * 2 // 64
NOMINAL_HBM_GBS = 7900.0


def nominal_peaks(device, peaks):
    """SMs x maximum SM clock x the per-SM bf16 rate, which the library's probe
    (back-to-back MMAs on one SM) measures here; the published HBM3e bandwidth."""
    import torch

    import ring_attention_online_gb300 as ra
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    mhz = float(peaks.get("sm_max_mhz", 2070.0))
    try:
        cpm = ra.attn_probe_mma_cycles(4096)
        rate, how = 128 * 128 * 16 * 2 / cpm, f"{cpm:.2f} cycles per 128x128x16 MMA, measured"
    except Exception as e:  # the probe is a diagnostic: keep the documented rate
        rate, how = float(BF16_FLOP_PER_CLK_PER_SM), f"probe failed ({e}); 64 cycles per MMA"
    return {"tflops": sms * rate * mhz * 1e6 / 1e12, "hbm_gbs": NOMINAL_HBM_GBS,
            "basis": f"{sms} SMs x {mhz:.0f} MHz x {rate:.0f} bf16 FLOP/clk/SM ({how}); HBM3e 7.9 TB/s"}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except OSError:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background (read-only)."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(r[1]) for r in rows]
        mx = [num(r[2]) for r in rows]
        power = [num(r[3]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        loaded = [s for s, p in zip(sm, power) if p == p and p > 200] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------ workloads (GPU side)
def causal_pairs(L: int) -> int:
    return L * (L + 1) // 2


def make_workload(name: str, device, batch=None, seq=None):
    """Inputs in HBM plus a step closure for one workload of the pages."""
    import torch

    import ring_attention_online_gb300 as ra
    import synthetic as syn
    cfg = dict(syn.WORKLOADS[name])
    if batch is not None:
        cfg["num_seqs" if cfg["kind"] == "jagged" else "B"] = batch
    if seq is not None and cfg["kind"] == "prefill":
        cfg["S_q"] = cfg["S_kv"] = seq
    w = {"name": name, "cfg": cfg}
    if cfg["kind"] == "prefill":
        q, k, v = syn.prefill_inputs(cfg, seed=0, device=device)
        o = torch.empty_like(q)
        lse = torch.empty(cfg["B"], cfg["h_q"], cfg["S_q"], device=device, dtype=torch.float32)
        C = cfg["num_chunks"]
        causal = cfg["causal"]
        window = cfg.get("window")

        def step(stream=None):
            if window is None:
                ra.attn_prefill(q, k, v, o, lse, causal=causal, num_chunks=C, stream=stream)
            else:
                ra.attn_prefill_window(q, k, v, o, lse, window=window, num_chunks=C, stream=stream)
        flops = 4.0 * cfg["D"] * cfg["B"] * cfg["h_q"] * causal_pairs(cfg["S_q"]) if causal else \
            4.0 * cfg["D"] * cfg["B"] * cfg["h_q"] * cfg["S_q"] * cfg["S_kv"]
        if window is not None:  # query i sees min(i, window) + 1 keys
            S = cfg["S_q"]
            pairs = window * (window + 1) // 2 + (S - window) * (window + 1) if S > window else S * (S + 1) // 2
            flops = 4.0 * cfg["D"] * cfg["B"] * cfg["h_q"] * pairs
        w.update(step=step, units=flops / 1e12, unit="TFLOP/s", bound="tensor", launches=1, tensors=(q, k, v, o, lse),
                 inputs=(q, k, v), outputs=(o, lse), kernel_units=flops / 1e12,
                 config=dict({"workload": name, "B": cfg["B"], "S": cfg["S_q"], "h_q": cfg["h_q"],
                              "h_kv": cfg["h_kv"], "D": cfg["D"], "causal": causal, "num_chunks": C,
                              "tile": "128x128", "l2": "inputs larger than L2 (no flush)"},
                             **({"window": window} if window is not None else {})))
        pipe = {}

        def e2e_step(host_in, host_out, stream):
            """One batch at a time through the public entry point, with the batches
            pipelined over three streams: batch b+1's inputs copy in while batch b
            computes and batch b-1's outputs copy out (the link runs both ways at
            once).  Events keep each batch's buffers from being overwritten before
            the previous step has used them.  Consecutive steps overlap too: a
            step's inputs start copying in once the previous step's kernels are
            enqueued, while its last outputs still copy out; the timed region
            ends after the last step's outputs are on the host (`e2e_finish`).
            Only the first step of a timed region holds its copies until the
            region's start (`e2e_begin`): later steps' copies are behind it anyway."""
            B = cfg["B"]
            if not pipe:
                pipe.update(h2d=torch.cuda.Stream(device), d2h=torch.cuda.Stream(device), started=False,
                            ev_in=[torch.cuda.Event() for _ in range(B)],
                            ev_c=[torch.cuda.Event() for _ in range(B)],
                            ev_out=[torch.cuda.Event() for _ in range(B)])
            h2d, d2h = pipe["h2d"], pipe["d2h"]
            if pipe.get("hold", True):
                pipe.setdefault("ev_start", torch.cuda.Event()).record(stream)
                h2d.wait_event(pipe["ev_start"])  # the copies start inside the timed region
                pipe["hold"] = False
            for b in range(B):
                if pipe["started"]:
                    h2d.wait_event(pipe["ev_c"][b])  # the previous step has read batch b's inputs
                with torch.cuda.stream(h2d):
                    for d, h in zip((q, k, v), host_in):
                        d[b].copy_(h[b], non_blocking=True)
                pipe["ev_in"][b].record(h2d)
                stream.wait_event(pipe["ev_in"][b])
                if pipe["started"]:
                    stream.wait_event(pipe["ev_out"][b])  # ... and copied out batch b's outputs
                sl = slice(b, b + 1)
                if window is None:
                    ra.attn_prefill(q[sl], k[sl], v[sl], o[sl], lse[sl], causal=causal, num_chunks=C, stream=stream)
                else:
                    ra.attn_prefill_window(q[sl], k[sl], v[sl], o[sl], lse[sl], window=window, num_chunks=C,
                                           stream=stream)
                pipe["ev_c"][b].record(stream)
                d2h.wait_event(pipe["ev_c"][b])
                with torch.cuda.stream(d2h):
                    for h, d in zip(host_out, (o, lse)):
                        h[b].copy_(d[b], non_blocking=True)
                pipe["ev_out"][b].record(d2h)
            pipe["started"] = True

        def e2e_begin():
            pipe["hold"] = True

        def e2e_finish(stream):
            stream.wait_event(pipe["ev_out"][cfg["B"] - 1])  # the last step's last output is on the host
        w["e2e_step"] = e2e_step
        w["e2e_begin"] = e2e_begin
        w["e2e_finish"] = e2e_finish
        w["e2e_launches"] = cfg["B"]  # one prefill kernel per batch
    elif cfg["kind"] == "jagged":
        q, k, v, offs = syn.jagged_inputs(cfg, seed=0, device=device)
        T = int(offs[-1])
        lens = offs[1:].astype("int64") - offs[:-1].astype("int64")
        max_len = int(lens.max())
        o = torch.empty_like(q)
        lse = torch.empty(cfg["H"], T, device=device, dtype=torch.float32)
        offs_d = torch.from_numpy(offs).to(device)
        ws = torch.empty(ra.attn_jagged_workspace_bytes(len(lens), T, max_len), dtype=torch.uint8, device=device)

        def step(stream=None):
            ra.attn_jagged(q, k, v, o, offs_d, max_len, ws, lse, causal=True, stream=stream)
        flops = 4.0 * cfg["D"] * cfg["H"] * float(sum(causal_pairs(int(L)) for L in lens))
        # Q, K, V read and O written once, plus the LSE: at 169 FLOP per byte this
        # workload sits below GB300's ridge point (measured bf16 / HBM peaks, ~288
        # FLOP per byte), so HBM is its binding roofline; the tensor fraction is
        # reported beside it
        hbm_bytes = 4.0 * T * cfg["H"] * cfg["D"] * 2 + cfg["H"] * T * 4.0
        # the worklist builder is one kernel up to 1024 sequences, a count and a
        # write kernel beyond; then the attention kernel
        launches = (1 if len(lens) <= 1024 else 2) + 1
        w.update(step=step, units=flops / 1e12, unit="TFLOP/s", bound="hbm", launches=launches, tensors=(q, k, v, o),
                 kernel_units=hbm_bytes / 1e9, tensor_units=flops / 1e12,
                 config={"workload": name, "num_seqs": cfg["num_seqs"], "total_tokens": T, "H": cfg["H"],
                         "D": cfg["D"], "len_range": [cfg["len_lo"], cfg["len_hi"]], "causal": True,
                         "l2": "inputs larger than L2 (no flush)"})
    else:  # decode
        q, k, v = syn.decode_inputs(cfg, seed=0, device=device)
        B, h_q, h_kv, D, S_kv, C = cfg["B"], cfg["h_q"], cfg["h_kv"], cfg["D"], cfg["S_kv"], cfg["num_splits"]
        o = torch.empty_like(q)
        lse = torch.empty(B, h_q, device=device, dtype=torch.float32)
        ws = torch.empty(ra.attn_decode_workspace_bytes(B, h_q, D, C), dtype=torch.uint8, device=device)
        rows = C * B * h_q

        def step(stream=None):  # one kernel: partials, and the fused merge in each group's last CTA
            ra.attn_decode_splitkv(q, k, v, o, ws, lse, num_splits=C, stream=stream)
        kv_bytes = 2.0 * B * S_kv * h_kv * D * 2
        part_bytes = rows * (D + 2) * 4.0
        alg_bytes = kv_bytes + q.numel() * 2 + part_bytes
        w.update(step=step, units=kv_bytes / 1e9, unit="GB/s", bound="hbm", launches=1, tensors=(q, k, v, o, ws),
                 kernel_units=alg_bytes / 1e9,
                 config={"workload": name, "B": B, "h_q": h_q, "h_kv": h_kv, "D": D, "S_kv": S_kv,
                         "num_splits": C, "l2": "inputs larger than L2 (no flush)",
                         "unit_note": "K+V bytes read once per step"})
    return w


def host_link(device, nbytes: int = 256 << 20, reps: int = 5):
    """Pinned host <-> device copy bandwidth (one cudaMemcpyAsync per copy), each
    direction alone and both at once on two streams, best of `reps`, with the
    host's NUMA layout: the ceiling of the end-to-end step."""
    import torch
    h = [torch.empty(nbytes, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    d = [torch.empty(nbytes, dtype=torch.uint8, device=device) for _ in range(2)]
    s = [torch.cuda.Stream(device) for _ in range(2)]

    def timed(fn):
        best = float("inf")
        for _ in range(reps + 1):  # the first run warms up
            torch.cuda.synchronize(device)
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize(device)
            best = min(best, time.perf_counter() - t0)
        return best

    def h2d():
        with torch.cuda.stream(s[0]):
            d[0].copy_(h[0], non_blocking=True)

    def d2h():
        with torch.cuda.stream(s[1]):
            h[1].copy_(d[1], non_blocking=True)

    def both():
        h2d()
        d2h()

    t_in, t_out, t_both = timed(h2d), timed(d2h), timed(both)
    try:
        nodes = open("/sys/devices/system/node/online").read().strip()
    except OSError:
        nodes = "unknown"
    cpus = sorted(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else []
    return {"h2d_gbs": round(nbytes / t_in / 1e9, 1), "d2h_gbs": round(nbytes / t_out / 1e9, 1),
            "both_gbs": round(2 * nbytes / t_both / 1e9, 1), "numa_nodes_online": nodes,
            "process_cpus": f"{cpus[0]}-{cpus[-1]} ({len(cpus)})" if cpus else "unknown",
            "how": "pinned torch tensors, one cudaMemcpyAsync per copy, 256 MiB, best of 5"}


def time_steps(step, K: int, W: int, device, finish=None, begin=None):
    """Device time of K steps after W warm-up steps.  `begin()`, if given, runs right
    after the start event is recorded; `finish(stream)` joins work the steps left on
    other streams into `stream` before the end event."""
    import torch
    stream = torch.cuda.current_stream(device)
    for _ in range(W):
        step(stream)
    torch.cuda.synchronize(device)
    barrier()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    if begin is not None:
        begin()
    for _ in range(K):
        step(stream)
    if finish is not None:
        finish(stream)
    end.record(stream)
    torch.cuda.synchronize(device)
    barrier()
    return start.elapsed_time(end)


def roofline(w, kernel_ms_per_launch: float, peaks, peak_kind: str, traffic=None, nominal=None):
    achieved = w["kernel_units"] / (kernel_ms_per_launch / 1e3)
    if w["bound"] == "tensor":
        peak, unit, nom = peaks["bf16_tflops"], "TFLOP/s", (nominal or {}).get("tflops")
    else:
        peak, unit, nom = peaks["hbm_gbs"], "GB/s", (nominal or {}).get("hbm_gbs")
    r = {"bound": w["bound"], "achieved": round(achieved, 2), "peak": peak, "unit": unit,
         "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": peak_kind}
    if nom:
        r["nominal"] = {"peak": round(nom, 1), "frac": round(achieved / nom, 4), "basis": nominal["basis"]}
    return r


def tensor_roofline(w, kernel_ms_per_launch: float, peaks, peak_kind: str, nominal=None):
    """The tensor-core fraction of a workload whose binding roofline is HBM."""
    if "tensor_units" not in w:
        return {}
    tfs = w["tensor_units"] / (kernel_ms_per_launch / 1e3)
    r = {"bound": "tensor", "achieved": round(tfs, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
         "frac": round(tfs / peaks["bf16_tflops"], 4), "peak_source": peak_kind}
    if nominal:
        r["nominal"] = {"peak": round(nominal["tflops"], 1), "frac": round(tfs / nominal["tflops"], 4),
                        "basis": nominal["basis"]}
    return {"roofline_tensor": r}


# ------------------------------------------------------------------ CPU legs (oracle)
def _cpu_slice():
    """One (batch, head) slice of the headline workload, drawn with its recipe (host)."""
    import torch
    cfg = __import__("synthetic").WORKLOADS[HEADLINE]
    S, D = cfg["S_q"], cfg["D"]
    gen = torch.Generator().manual_seed(0)
    return tuple(torch.randn(1, S, 1, D, generator=gen).bfloat16() for _ in range(3))


def cpu_sample_dense(seconds: float, rows_per_sample: int = 512, qkv=None, first_block: int = 0,
                     max_blocks: int | None = None):
    """fp64 oracle on query-row blocks of one (batch, head) slice of the headline
    workload (host cores); the slice is drawn before the clock starts.  Blocks are
    taken with a stride of 13 blocks (coprime with the block count), so that a few
    blocks already mix short and long causal rows."""
    import numpy as np

    from oracle import attention as A
    cfg = __import__("synthetic").WORKLOADS[HEADLINE]
    S, D = cfg["S_q"], cfg["D"]
    q, k, v = qkv if qkv is not None else _cpu_slice()
    flops = 0.0
    n = 0
    t0 = time.perf_counter()
    while max_blocks is None or n < max_blocks:
        n_blocks = (S + rows_per_sample - 1) // rows_per_sample
        lo = (((first_block + n) * 13) % n_blocks) * rows_per_sample
        rows = np.arange(lo, min(S, lo + rows_per_sample))
        A.attention(q, k, v, 1 / math.sqrt(D), True, rows=rows)
        flops += 4.0 * D * float(np.sum(rows + 1))
        n += 1
        el = time.perf_counter() - t0
        if max_blocks is None and el >= seconds:
            break
    return flops, time.perf_counter() - t0, n


def cpu_baseline(seconds: float = 15.0):
    flops, el, n = cpu_sample_dense(seconds)
    return {"value": round(flops / el / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} blocks of 512 query rows x all visible keys of one (batch, head) of {HEADLINE} "
                      f"(fp64 NumPy, {el:.1f} s)"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    W, K = args.warmup, args.steps
    # each step: the next block of 128 query rows of one (batch, head) against all
    # their visible keys (bounded work, blocks in the stride-13 order of
    # cpu_sample_dense); the slice is drawn before the clock starts
    qkv = _cpu_slice()
    cpu_sample_dense(0.0, 128, qkv, 0, min(W, 1))
    flops, el, _ = cpu_sample_dense(0.0, 128, qkv, 0, K)
    value = flops / el / 1e12
    line = {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": K,
            "warmup": W, "ms_per_step": round(el * 1e3 / K, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": HEADLINE, "B": 8, "S": 4096, "h_q": 32, "h_kv": 32, "D": 256, "causal": True,
                       "sample_per_step": "128 query rows x visible keys of one (batch, head)"},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{K} steps, each a block of 128 query rows of one (batch, head) "
                                       f"against all their visible keys, fp64 NumPy"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ main (GPU)
def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        init_dist(world, "nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    import ring_attention_online_gb300 as ra
    ra.load_library()
    peaks, peak_kind = load_peaks()
    nominal = nominal_peaks(device, peaks)
    K, W = args.steps, max(args.warmup, 3)

    # ---- headline (or the workload named on the command line)
    w = make_workload(args.workload, device, args.batch, args.seq)
    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    clocks = ClockSampler(int(visible[local]) if len(visible) > local and visible[local].isdigit() else local)
    for _ in range(W):
        w["step"]()
    torch.cuda.synchronize(device)
    clocks.start()
    time.sleep(0.2)
    ms = time_steps(w["step"], K, 1, device)
    clk = clocks.stop()
    units, ms_max = aggregate(w["units"] * K, ms, world, device)
    status = ra.attn_last_device_status()
    if status != 0:
        raise RuntimeError(f"device status {ra.STATUS.get(status)} after the headline run")
    value = units / (ms_max / 1e3)
    kernel_ms = ms / K  # the dominant kernel's share of a step
    traffic = _profiled_traffic(args.workload) if args.batch is None and args.seq is None else None
    line = {"metric": METRIC, "value": round(value, 2), "unit": w["unit"], "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": round(ms_max / K, 4), "higher_is_better": True, "scaling": "weak",
            # the pages' figure is another machine's, at unstated precision: context, not a baseline
            "vs_baseline": None,
            "pages_context_ratio": round(value / world / PAGES_DENSE_CAUSAL_TFS, 3) if args.workload == HEADLINE and
            args.batch is None and args.seq is None else None, "dtype": "bf16", "data": "synthetic",
            "config": dict(w["config"], parallelism=f"replicas{world}" if world > 1 else "single"),
            "roofline": roofline(w, kernel_ms, peaks, peak_kind, traffic, nominal),
            **tensor_roofline(w, kernel_ms, peaks, peak_kind, nominal),
            "gpu_launches": K * w["launches"],
            "clocks": clk}

    # ---- end to end through the public API with host buffers
    if not args.no_e2e and "e2e_step" in w:
        host_in = [t.detach().cpu().pin_memory() for t in w["inputs"]]
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in w["outputs"]]
        stream = torch.cuda.current_stream(device)
        e2e_step = lambda s=None: w["e2e_step"](host_in, host_out, stream)  # noqa: E731
        K2 = max(3, K // 5)
        ms_e2e = time_steps(e2e_step, K2, 2, device, finish=w.get("e2e_finish"), begin=w.get("e2e_begin"))
        units_e2e, ms_e2e_max = aggregate(w["units"] * K2, ms_e2e, world, device)
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out)
        e2e_launches = K2 * w.get("e2e_launches", w["launches"])
        line["e2e"] = {"value": round(units_e2e / (ms_e2e_max / 1e3), 2), "unit": w["unit"],
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K2,
                       "gpu_launches": e2e_launches}
        # the step's copies can take no less than the link allows: all inputs in one
        # direction, all outputs in the other, and both together on the shared link
        link = host_link(device)
        floor_ms = 1e3 * max(h2d / (link["h2d_gbs"] * 1e9), d2h / (link["d2h_gbs"] * 1e9),
                             (h2d + d2h) / (link["both_gbs"] * 1e9))
        link["step_floor_ms"] = round(floor_ms, 3)
        link["e2e_ms_per_step"] = round(ms_e2e_max / K2, 3)
        link["e2e_frac_of_link_floor"] = round(floor_ms / (ms_e2e_max / K2), 3)
        line["e2e"]["host_link"] = link
        line["gpu_launches"] += e2e_launches
        del host_in, host_out
    del w
    torch.cuda.empty_cache()

    # ---- secondary workloads (same rules: inputs in HBM, CUDA events, max over ranks)
    if not args.no_secondary and args.workload == HEADLINE and args.batch is None and args.seq is None:
        sec = []
        for name in SECONDARY:
            w = make_workload(name, device)
            k2 = max(3, min(K, 20))
            ms2 = time_steps(w["step"], k2, W, device)
            units2, ms2_max = aggregate(w["units"] * k2, ms2, world, device)
            kernel_ms = ms2 / k2
            entry = {"workload": name, "value": round(units2 / (ms2_max / 1e3), 2), "unit": w["unit"],
                     "ms_per_step": round(ms2_max / k2, 4), "steps": k2, "config": w["config"],
                     "roofline": roofline(w, kernel_ms, peaks, peak_kind, _profiled_traffic(name), nominal)}
            entry.update(tensor_roofline(w, kernel_ms, peaks, peak_kind, nominal))
            sec.append(entry)
            line["gpu_launches"] += k2 * w["launches"]
            status = ra.attn_last_device_status()
            if status != 0:
                raise RuntimeError(f"device status {ra.STATUS.get(status)} after {name}")
            del w
            torch.cuda.empty_cache()
        line["secondary"] = sec

    # ---- CPU baseline: the oracle on host cores (rank 0, N = 1 only)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == HEADLINE:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def _profiled_traffic(name: str):
    """DRAM bytes per launch of the workload's dominant kernel from the committed ncu summary, if any."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            return json.load(f).get(name)
    except (OSError, ValueError):
        return None


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
