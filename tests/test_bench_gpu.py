"""The benchmark's output: one JSON line whose keys and figures agree with one another.

Runs `bench.py` on the prefill workload with a few steps and no extra tables, as a
separate process (as a user would), and checks the measurement contract: the metric's
units, throughput equal to tokens over the step time, the roofline fraction equal to
achieved over peak, the end-to-end leg's copied bytes, one kernel launch per timed
step, and the clock record.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
T, H = 4096, 2048


def _bench(*args):
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    return json.loads(lines[0])


def test_prefill_line_keeps_the_contract():
    steps, warmup = 5, 3
    d = _bench("--steps", str(steps), "--warmup", str(warmup), "--no-extra", "--no-cpu-baseline")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["dtype"] == "bf16" and d["vs_baseline"] is None
    assert d["config"]["workload"] == "qwen3_30b_a3b_moe_prefill_T4096_zipf1.2"
    assert d["config"]["tokens_per_gpu"] == T
    # tokens/s x seconds per step = the tokens of one step
    assert d["value"] > 0
    assert abs(d["value"] * d["ms_per_step"] / 1e3 - T) <= 1e-6 * T
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s"
    assert abs(rf["achieved"] / rf["peak"] - rf["frac"]) <= 1e-9
    assert 0.05 < rf["frac"] < 1.5
    # achieved = the layer's algorithmic FLOP / the measured step time
    assert abs(rf["algorithmic_flops_per_launch"] / (d["ms_per_step"] / 1e3) / 1e12
               - rf["achieved"]) <= 1e-6 * rf["achieved"]
    e2e = d["e2e"]
    assert e2e["unit"] == "tokens/s" and e2e["value"] > 0
    assert e2e["h2d_bytes_per_step"] == T * H * 2   # bf16 x
    assert e2e["d2h_bytes_per_step"] == T * H * 4   # fp32 out
    assert d["gpu_launches"] == steps                # one megakernel per layer call
    assert d["clocks"] is None or "sm_mhz" in d["clocks"]
