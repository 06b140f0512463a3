"""The benchmark's output contract on a GPU: one JSON line with the metric, the timing
fields, the roofline object, the end-to-end figure, the launch count and the clock
record, from a short run of bench.py (no sweep, no CPU baseline)."""
from __future__ import annotations

import json
import subprocess
import sys
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu
ROOT = Path(__file__).resolve().parents[1]


def test_bench_prints_one_json_line_with_the_contract_keys():
    steps, warmup = 20, 3                   # not a multiple of the graph length
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--steps", str(steps),
                        "--warmup", str(warmup), "--no-sweep", "--no-cpu-baseline",
                        "--e2e-steps", "10"], capture_output=True, text=True, cwd=ROOT,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-4000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == steps        # exactly the requested steps
    t = d["timing"]
    assert t["steps_per_region"] == steps and t["regions"] >= 3
    assert t["min_ms"] <= t["median_ms"] <= t["max_ms"] and t["timed_region_s"] >= 0.25
    assert abs(d["ms_per_step"] * steps - t["median_ms"]) < 1e-9
    assert d["clocks"]["samples"] >= 3 and "shorter" not in d["clocks"]["note"]
    assert d["warmup"] == warmup and d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["config"]["workload"] == "roundtrip_v41_16384"
    # value = tokens per step / seconds per step
    assert abs(d["value"] * d["ms_per_step"] * 1e-3 / d["config"]["tokens"] - 1) < 1e-6
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9 and 0 < rf["frac"] < 1.5
    assert rf["traffic"] is None or rf["traffic"] > 0
    assert rf["stream_same_bytes"]["gbs"] > 0
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == "tokens/s"
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] == 16384 * 1024
    assert e["value"] < d["value"]                       # host copies inside the step
    assert d["gpu_launches"] == 2 * d["steps"]
    em = d["early_metadata"]
    assert em["value"] > 0 and abs(em["value"] * em["ms_per_step"] * 1e-3 / 16384 - 1) < 1e-6
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    for k in ("insert", "gather"):
        kk = d["kernels"][k]
        assert kk["us"] > 0 and kk["after_l2_flush_us"] > 0 and kk["alg_bytes"] > 0
    assert "sweep" not in d and "cpu_baseline" not in d
