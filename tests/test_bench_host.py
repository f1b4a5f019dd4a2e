"""Host-side pieces of bench.py that need no GPU: the reference arm's step plan,
the host description beside the oracle timing, and the rule that a recorded
DRAM-traffic figure is reported only while the kernel source it was taken from
is unchanged."""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("steps,warmup", [(500, 5), (20, 3), (3, 1), (1, 0), (10000, 10)])
def test_reference_plan_stays_within_budget(steps, warmup):
    per_step, n = bench.reference_plan(steps, warmup)
    assert per_step >= bench.STEP_MIN_S
    assert 1 <= n <= steps
    # the planned run fits the budget unless a single timed step already needs more
    assert (warmup + n) * per_step <= bench.REF_BUDGET_S + 1e-9 or n == 1
    if (steps + warmup) * bench.STEP_MIN_S <= bench.REF_BUDGET_S:
        assert n == steps   # nothing cut when the asked-for steps fit


def test_host_cpu_reports_machine_and_cores():
    h = bench.host_cpu()
    assert h["machine"] and h["nproc"] >= 1


def _traffic_root(tmp_path, src_text, recorded_src_text):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "k.cu").write_text(src_text)
    rec = {"kern": {"workload": "w", "dram_bytes_per_launch": 123,
                    "source_sha256_16": hashlib.sha256(recorded_src_text.encode()).hexdigest()[:16],
                    "sources": ["k.cu"]}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    return str(tmp_path)


def test_recorded_traffic_only_for_the_captured_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", _traffic_root(tmp_path, "int a;", "int a;"))
    assert bench.recorded_traffic("kern", "w") == 123
    assert bench.recorded_traffic("kern", "other workload") is None
    assert bench.recorded_traffic("other kernel", "w") is None


def test_recorded_traffic_dropped_after_a_source_change(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", _traffic_root(tmp_path, "int a; // edited", "int a;"))
    assert bench.recorded_traffic("kern", "w") is None


def test_recorded_traffic_per_workload_key(tmp_path, monkeypatch):
    """A second capture of the same kernel on another workload lives under
    "<kernel> @ <workload>"; the plain key keeps serving its own workload."""
    root = _traffic_root(tmp_path, "int a;", "int a;")
    p = tmp_path / "profiles" / "traffic.json"
    rec = json.loads(p.read_text())
    rec["kern @ w2"] = dict(rec["kern"], workload="w2", dram_bytes_per_launch=456)
    p.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", root)
    assert bench.recorded_traffic("kern", "w") == 123
    assert bench.recorded_traffic("kern", "w2") == 456
    assert bench.recorded_traffic("kern", "w3") is None

