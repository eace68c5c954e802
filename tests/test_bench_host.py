"""bench.py host logic on CPU: clock-sample summary, the source-hash gate on recorded DRAM
traffic, and the reference arm's JSON line (the float64 oracle timed on host cores)."""

import json
import os
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_clock_samples_median_max_and_reasons():
    rows = [
        "2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n",
        "1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active\n",
        "2070, 2070, 1200.5, 0x0, Not Active, Not Active, Not Active, Not Active\n",
        "[N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active\n",   # unparsable: skipped
        "\n",
    ]
    got = bench.summarize_clock_samples(rows)
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    hot = ["1500, 2070, 1400, 0x40, Not Active, Active, Active, Not Active\n"]
    assert bench.summarize_clock_samples(hot)["reasons"] == ["hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert bench.summarize_clock_samples([]) is None


def _profile(tmp_path, workload, sha, traffic):
    d = tmp_path / "profiles"
    d.mkdir(exist_ok=True)
    (d / f"{workload}.md").write_text(f"# summary\n\nworkload: {workload}\n\ntraffic_bytes_per_launch: {traffic}\n"
                                      f"kernel_source_sha256: {sha}\n")


def test_recorded_traffic_only_while_kernel_sources_hash_the_same(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda cfg: "abc123")
    _profile(tmp_path, "batched_paged", "abc123", 1167529216)
    _profile(tmp_path, "long_context", "stale0", 538345728)
    assert bench.recorded_traffic("batched_paged") == 1167529216
    assert bench.recorded_traffic("long_context") is None      # the kernels changed since the capture
    assert bench.recorded_traffic("prefill_128k") is None      # no capture at all
    assert bench.recorded_traffic("no_such_workload") is None


def test_committed_profiles_name_known_workloads():
    """Every committed ncu summary with a launch list names a workload of the bench, once, and
    carries the traffic and source-hash lines the bench reads."""
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "profiles"))):
        text = open(os.path.join(ROOT, "profiles", fn), encoding="utf-8").read()
        lines = {ln.split(":", 1)[0]: ln.split(":", 1)[1].strip() for ln in text.splitlines()
                 if ln.startswith(("workload:", "traffic_bytes_per_launch:", "kernel_source_sha256:"))}
        if not lines:          # a single-kernel summary without a launch list
            continue
        assert lines.get("workload") in bench.CONFIGS, fn
        assert int(lines["traffic_bytes_per_launch"]) > 0, fn
        assert len(lines["kernel_source_sha256"]) == 16, fn
        names.append(lines["workload"])
    assert len(names) == len(set(names)) >= 9


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    d = json.loads(lines[-1])
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["unit"] == "GB/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "batched_paged"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
