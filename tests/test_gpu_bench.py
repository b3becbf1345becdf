"""bench.py's JSON line on a GPU: the fields the measurement record carries
(workload, roofline, CPU baseline, end to end, launch count, clocks) and
their consistency with one another, from a short run of the script itself."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
B, GAMMA, V = 64, 16, 131072  # the block-diffusion workload the script times


def test_bench_line_carries_the_measurement_fields():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "4", "--warmup", "3"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 4 and d["warmup"] >= 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["data"] == "synthetic"
    # value: verified rows (B * gamma per call) over the timed time per call
    assert d["value"] > 0
    assert abs(d["value"] - B * GAMMA / (d["ms_per_step"] / 1e3)) <= 1e-9 * d["value"]
    assert "workload" in d["config"]

    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["kernel"] == "k_row_stats"
    assert rf["algorithmic_bytes_per_launch"] == B * (2 * GAMMA + 1) * V * 2
    assert abs(rf["achieved"] - rf["algorithmic_bytes_per_launch"] / (rf["avg_launch_ms"] / 1e3) / 1e9) \
        <= 1e-9 * rf["achieved"]
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) <= 1e-12 and 0.3 < rf["frac"] < 1.2
    assert rf["traffic"] is None or rf["traffic"] > rf["algorithmic_bytes_per_launch"] * 0.99
    # the kernel's own events lie inside the call, so it cannot take longer than a call
    assert rf["avg_launch_ms"] < d["ms_per_step"] * 1.2

    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]
    assert cb["unit"] == d["unit"]

    e = d["e2e"]
    assert e["unit"] == d["unit"] and e["value"] > 0
    assert e["h2d_bytes_per_step"] >= B * (2 * GAMMA + 1) * V * 2  # the logits cross the link every step
    assert e["d2h_bytes_per_step"] >= B * 4  # at least the accept lengths come back

    assert d["gpu_launches"] == 2 * d["steps"]  # streaming + finish kernel per call
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
