"""The reference arm of bench.py (the CPU oracle timed on the host cores)
prints one JSON line with the keys a bench line carries; it needs no GPU."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.strip().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["unit"] == "tok/s" and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0
    # a step is one token through the 48 layers (batch 1): tok/s = 1 / seconds per step
    assert abs(d["value"] - 1.0 / (d["ms_per_step"] * 1e-3)) <= 0.01 * d["value"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("decode48")


def test_reported_miss_rate_bound_is_the_pages_arithmetic():
    """bench.py's max_miss_rate_for_rate is the oracle's bound: with the
    pages' worked numbers (50 GB/s, 87.7 tok/s, 48 layers, top-8, the 4.72 MB
    block-FP8 expert) both give the pages' 31 %."""
    import importlib.util

    from oracle import sizing

    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    fp8 = sizing.expert_bytes(2048, 768, "fp8")
    got = bench.max_miss_rate_for_rate(50.0, 87.7, 48, 8, fp8)
    assert abs(got - sizing.max_miss_rate(50e9, 87.7, 48, 8, fp8)) < 1e-12
    assert round(got, 2) == 0.31
