"""bench.py host logic on CPU: max-over-ranks aggregation with two gloo ranks,
and the reference arm (the fp64 oracle on host cores) end to end."""

import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    units, ms = bench.aggregate(per_rank_units=10.0, per_rank_ms=5.0 + 3.0 * rank, world=world)
    bench.barrier()
    out[rank] = (units, ms)
    dist.destroy_process_group()


def test_aggregate_takes_max_time_over_two_gloo_ranks():
    port = 29500 + os.getpid() % 1000
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1] == (20.0, 8.0)


def test_aggregate_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(3.0, 7.5, 1) == (3.0, 7.5)


def _run_bench(args, env_extra=None):
    env = dict(os.environ, **(env_extra or {}))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          env=env, timeout=600, cwd=ROOT)


def test_reference_arm_prints_one_contract_line():
    r = _run_bench(["--impl", "reference", "--steps", "2", "--warmup", "1"])
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["config"]["workload"] == "dense_causal_b8_h32_s4096_d256"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_nonzero_rank_is_silent():
    r = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "1"], {"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_every_reported_workload_has_profiled_traffic():
    """The roofline objects of the headline and of every secondary workload carry the DRAM
    bytes per launch committed under profiles/ (traffic.json), not null."""
    sys.path.insert(0, ROOT)
    import bench
    import synthetic as syn
    for name in (bench.HEADLINE,) + bench.SECONDARY:
        assert name in syn.WORKLOADS
        t = bench._profiled_traffic(name)
        assert isinstance(t, int) and t > 0, name


def test_roofline_objects():
    """Achieved = algorithmic units per launch / launch time; a workload bound by HBM
    (below the ridge point) reports its tensor fraction beside the binding roofline."""
    sys.path.insert(0, ROOT)
    import bench
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0}
    dense = {"bound": "tensor", "kernel_units": 0.55}  # TFLOP per launch
    r = bench.roofline(dense, 0.5, peaks, "measured", traffic=123)
    assert r == {"bound": "tensor", "achieved": 1100.0, "peak": 2000.0, "unit": "TFLOP/s", "frac": 0.55,
                 "traffic": 123, "peak_source": "measured"}
    assert bench.tensor_roofline(dense, 0.5, peaks, "measured") == {}
    jag = {"bound": "hbm", "kernel_units": 2.4, "tensor_units": 0.45}  # GB and TFLOP per launch
    r = bench.roofline(jag, 0.8, peaks, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["achieved"] == 3000.0 and r["frac"] == 0.5
    t = bench.tensor_roofline(jag, 0.8, peaks, "measured")["roofline_tensor"]
    assert t["achieved"] == 562.5 and t["frac"] == 0.2812 and t["unit"] == "TFLOP/s"
    # nominal denominators beside the measured ones
    nom = {"tflops": 2500.0, "hbm_gbs": 8000.0, "basis": "test"}
    assert bench.roofline(dense, 0.5, peaks, "measured", nominal=nom)["nominal"] == {"peak": 2500.0, "frac": 0.44,
                                                                                     "basis": "test"}
    assert bench.roofline(jag, 0.8, peaks, "measured", nominal=nom)["nominal"]["frac"] == 0.375
    assert bench.tensor_roofline(jag, 0.8, peaks, "measured", nom)["roofline_tensor"]["nominal"]["frac"] == 0.225
    assert bench.BF16_FLOP_PER_CLK_PER_SM == 8192
