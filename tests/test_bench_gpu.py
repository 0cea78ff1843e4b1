"""bench.py's GPU arm prints the one JSON line the benchmark contract asks for:
whole-job throughput of the sweep step, the end-to-end figure through the C
ABI with host buffers, the roofline of the dominant kernel against the
measured peak, parity statistics, clocks and the launch count.  A short run
(two timed steps, no extra measurements, no CPU baseline)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_keys_and_consistency():
    env = dict(os.environ)
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "2",
                        "--warmup", "3", "--skip-extra", "--no-cpu-baseline"],
                       capture_output=True, text=True, cwd=ROOT, env=env, timeout=1200)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, lines
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e",
                "gpu_launches", "roofline", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True and d["value"] > 0
    assert "workload" in d["config"]
    # value is the step's FLOPs (2mnk over the 36 shapes) over its time
    flops = sum(2.0 * s["m"] * s["n"] * s["k"] for s in d["shapes"])
    assert d["value"] == pytest.approx(flops / (d["ms_per_step"] * 1e-3) / 1e12, rel=1e-3)
    e2e = d["e2e"]
    assert e2e["unit"] == d["unit"] and 0 < e2e["value"] < d["value"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    link = e2e["host_link"]
    assert link["h2d_GBps"] > 0 and link["d2h_GBps"] > 0 and link["both_GBps"] > 0
    # the transfers alone cannot take longer than the measured step
    assert link["transfer_bound_ms_per_step"] <= e2e["ms_per_step"] * 1.05
    assert d["gpu_launches"] == 2 * len(d["shapes"]) * d["steps"]
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s"
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"], rel=1e-3)
    assert 0 < rf["frac"] < 1.2
    # every shape's parity against the oracle within the gate
    assert len(d["shapes"]) == 36
    for s in d["shapes"]:
        assert s["max_norm_err"] <= 2e-3 and s["calc_diff"] < 1e-4, s
    assert "sm_mhz" in d["clocks"]
