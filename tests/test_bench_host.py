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


def _traffic(tmp_path, records):
    d = tmp_path / "profiles"
    d.mkdir(exist_ok=True)
    (d / "traffic.json").write_text(json.dumps(records))


def test_recorded_traffic_only_while_kernel_sources_hash_the_same(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda cfg: "abc123")
    _traffic(tmp_path, {"batched_paged": {"traffic_bytes_per_launch": 1167529216, "kernel_source_sha256": "abc123"},
                        "long_context": {"traffic_bytes_per_launch": 538345728, "kernel_source_sha256": "stale0"}})
    assert bench.recorded_traffic("batched_paged") == 1167529216
    assert bench.recorded_traffic("long_context") is None      # the kernels changed since the capture
    assert bench.recorded_traffic("prefill_128k") is None      # no capture at all
    assert bench.recorded_traffic("no_such_workload") is None


def test_recorded_traffic_without_a_data_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("batched_paged") is None


def test_committed_traffic_records_name_known_workloads_and_summaries():
    """Every record of the committed traffic file names a bench workload, a positive byte count,
    a 16-hex-digit source hash and an ncu summary under profiles/ that exists."""
    with open(os.path.join(ROOT, "profiles", "traffic.json"), encoding="utf-8") as f:
        recs = json.load(f)
    assert len(recs) >= 9
    for name, rec in recs.items():
        assert name in bench.CONFIGS, name
        assert isinstance(rec["traffic_bytes_per_launch"], int) and rec["traffic_bytes_per_launch"] > 0, name
        assert len(rec["kernel_source_sha256"]) == 16, name
        assert rec["summary"].startswith("profiles/") and os.path.exists(os.path.join(ROOT, rec["summary"])), name


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


def test_default_run_adds_the_long_context_record():
    """With no --workload the bench measures batched_paged and adds a long_context record (its own
    timing, roofline, clocks and e2e); the keys that describe the whole line are not repeated."""
    args = bench.parse_args([])
    assert args.workload is None and not args.no_extra
    assert bench.workload_config(args).name == bench.DEFAULT_WORKLOAD == "batched_paged"
    assert bench.EXTRA_WORKLOAD == "long_context" and bench.CONFIGS["long_context"].num_splits == 128
    for k in ("value", "ms_per_step", "roofline", "clocks", "e2e", "config", "gpu_launches"):
        assert k not in bench.SHARED_KEYS
    assert bench.parse_args(["--workload", "batched_paged"]).workload == "batched_paged"


def test_cpu_worker_reports_all_cores_and_one_core():
    r = subprocess.run([sys.executable, "bench.py", "--cpu-worker", "--cpu-seconds", "0.5"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["kind"] == "oracle" and d["value"] > 0 and d["unit"] == "GB/s"
    assert 1 <= d["cores"] <= bench.host_cores()
    assert d["one_core"]["cores"] == 1 and d["one_core"]["value"] > 0
