"""Host logic of bench.py that needs no GPU: the reference arm's JSON line, the
rule that a recorded DRAM-traffic figure counts only for the kernel source it
was measured on, and the thread count reported beside the CPU baseline."""
import hashlib
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny_f32", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr
    lines = [line for line in r.stdout.splitlines() if line.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["impl"] == "reference" and j["metric"] == bench.METRIC and j["unit"] == bench.UNIT
    assert j["value"] > 0 and j["steps"] == 1 and j["warmup"] == 1 and j["higher_is_better"]
    assert j["ms_per_step"] == pytest.approx(1e3 * synth.CONFIGS["tiny_f32"].T / j["value"])
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == j["value"] and cb["cores"] >= 1 and cb["sample"]
    assert j["e2e"] == {"value": j["value"], "unit": j["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert j["config"]["workload"].startswith("tiny_f32:")


def _fake_tree(tmp_path, source_text, recorded_hash):
    src_dir = tmp_path / "combine_top_route_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (src_dir / "k.cu").write_bytes(source_text)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"wl": {"kern": {"source": "k.cu", "source_sha256_16": recorded_hash,
                         "bytes_per_launch": 12345}}}))


def test_recorded_traffic_counts_only_for_the_measured_source(tmp_path, monkeypatch):
    text = b"__global__ void k() {}\n"
    _fake_tree(tmp_path, text, hashlib.sha256(text).hexdigest()[:16])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("wl", "kern") == 12345
    assert bench.recorded_traffic("wl", "other") is None
    assert bench.recorded_traffic("other", "kern") is None
    # the kernel source changed since the capture: no figure
    (tmp_path / "combine_top_route_gb300" / "csrc" / "k.cu").write_bytes(text + b"// edit\n")
    assert bench.recorded_traffic("wl", "kern") is None


def test_recorded_traffic_without_a_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("olmoe_fwd", "expert_up") is None


def test_committed_traffic_entries_name_existing_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        j = json.load(f)
    for wl, kernels in j.items():
        if wl.startswith("_"):
            continue
        assert wl.split(":")[0] in synth.CONFIGS, wl
        for e in kernels.values():
            assert os.path.exists(os.path.join(ROOT, "combine_top_route_gb300", "csrc", e["source"]))
            assert e["bytes_per_launch"] > 0 and len(e["source_sha256_16"]) == 16


def test_thread_caps_set_the_reported_cores(monkeypatch):
    for k in bench.THREAD_ENV:
        monkeypatch.delenv(k, raising=False)
    monkeypatch.setenv("OPENBLAS_NUM_THREADS", "1")
    o = bench.OracleSample(synth.CONFIGS["tiny_f32"])
    assert o.cores == 1
    assert o.run(32) > 0


def test_one_core_baseline_runs_in_a_capped_child():
    r = bench.cpu_baseline_one_thread(synth.CONFIGS["tiny_f32"], 0.5)
    assert "error" not in r, r
    assert r["cores"] == 1 and r["kind"] == "oracle" and r["value"] > 0
