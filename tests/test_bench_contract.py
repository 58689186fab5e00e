"""The benchmark's JSON line on the host: the reference arm (the CPU oracle on
a bounded sample) prints the contract's keys, and the DRAM traffic it carries
for the GPU arm comes only from a record taken on the current kernel sources
with the same launch plan."""
import importlib.util
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod_c", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "96x80x64:rr:hf", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    assert line["value"] > 0 and line["dtype"] == "f64" and line["unit"] == "TFLOP/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert (line["config"]["M"], line["config"]["N"], line["config"]["K"]) == (96, 80, 64)


def test_recorded_traffic_needs_current_sources_and_plan(tmp_path, monkeypatch):
    b = _bench()
    csrc = tmp_path / "dense_gemm_tmem_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cuh").write_text("kernel v1")
    (tmp_path / "profiles").mkdir()
    plan = {k: 1 for k in b.TRAFFIC_PLAN_KEYS}
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    rec = {"w": {"sources": ["k.cuh"], "src_hash": b.kernel_source_hash(["k.cuh"]),
                 "plan": dict(plan), "dram_bytes_per_launch": 123.0}}
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(rec))
    assert b.recorded_traffic("w", plan) == 123.0
    assert b.recorded_traffic("other", plan) is None
    changed = dict(plan)
    changed["k_group"] = 2  # another launch configuration
    assert b.recorded_traffic("w", changed) is None
    (csrc / "k.cuh").write_text("kernel v2")  # the kernel changed since the capture
    assert b.recorded_traffic("w", plan) is None


def test_committed_traffic_records_name_their_command():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        recs = json.load(f)
    b = _bench()
    for name, rec in recs.items():
        assert set(rec["plan"]) == set(b.TRAFFIC_PLAN_KEYS), name
        assert rec["command"].startswith("ncu ") and "--clock-control none" in rec["command"], name
        assert rec["dram_bytes_per_launch"] == pytest.approx(
            rec["dram_read_bytes"] + rec["dram_write_bytes"]), name
