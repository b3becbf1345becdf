"""Host logic of bench.py that needs no GPU: the clock-sample summary, the
traffic figure's link to the kernel source, the peak lookup, and the JSON
line of the reference arm (the oracle on the host cores)."""
import io
import json
import os
from contextlib import redirect_stdout

import bench


def test_clock_summary_parses_samples():
    c = bench.ClockSampler(0)
    c.lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2055, 2070, 1100.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1200.0, 0x8, Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = c.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    empty = bench.ClockSampler(0).summary()
    assert empty["samples"] == 0 and empty["sm_mhz"] is None


def test_traffic_is_reported_only_for_the_profiled_source(tmp_path, monkeypatch):
    good = tmp_path / "good.json"
    good.write_text(json.dumps({"kernel_source_sha": bench.kernel_source_hash(),
                                "traffic_bytes_per_launch": 123456}))
    stale = tmp_path / "stale.json"
    stale.write_text(json.dumps({"kernel_source_sha": "0000000000000000", "traffic_bytes_per_launch": 123456}))
    bad = tmp_path / "bad.json"
    bad.write_text("kernel_source_sha: not json")
    monkeypatch.setattr(bench, "PROFILE_RECORD", str(good))
    assert bench.profiled_traffic() == 123456.0
    for f in (stale, bad, tmp_path / "missing.json"):
        monkeypatch.setattr(bench, "PROFILE_RECORD", str(f))
        assert bench.profiled_traffic() is None


def test_product_arm_does_not_load_the_oracle():
    """Only the CPU-baseline and reference legs may load the oracle: bench.py
    itself imports neither it nor the test helpers at module level, and the
    product arm's functions take their inputs from the generator module."""
    import ast
    src = open(bench.__file__).read()
    tree = ast.parse(src)
    top = [n for n in tree.body if isinstance(n, (ast.Import, ast.ImportFrom))]
    names = {a.name for n in top for a in n.names} | {getattr(n, "module", None) for n in top}
    assert "oracle" not in names and "tests" not in names
    assert "_helpers" not in src
    for fn in tree.body:
        if isinstance(fn, ast.FunctionDef) and fn.name not in ("time_oracle",):
            for n in ast.walk(fn):
                if isinstance(n, ast.Import):
                    assert all(a.name != "oracle" for a in n.names), fn.name


def test_kernel_source_hash_follows_the_sources(tmp_path, monkeypatch):
    a, b = tmp_path / "a.cuh", tmp_path / "b.cuh"
    a.write_text("one")
    b.write_text("two")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", ["a.cuh", "b.cuh"])
    h0 = bench.kernel_source_hash()
    assert h0 == bench.kernel_source_hash()
    b.write_text("two!")
    assert bench.kernel_source_hash() != h0


def test_peak_lookup(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peak_gbs() == (6800.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6771.1}))
    assert bench.measured_peak_gbs() == (6771.1, "measured")


def test_reference_arm_prints_one_json_line(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    lines = [l for l in buf.getvalue().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 1
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == (os.cpu_count() or 1) and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith(bench.WORKLOAD)
