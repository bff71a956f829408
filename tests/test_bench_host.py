"""Host logic of bench.py that needs no GPU: the clock sampler's parsing of
nvidia-smi output (median SM clock under load, the throttle reasons seen),
driven by a stand-in nvidia-smi on PATH; the measured-peaks lookup; and the
workload description in the JSON line."""
import json
import os
import stat
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _fake_smi(tmp_path, lines):
    script = tmp_path / "nvidia-smi"
    body = "\n".join(f"echo '{ln}'" for ln in lines)
    script.write_text(f"#!/bin/sh\n{body}\nexec sleep 30\n")
    script.chmod(script.stat().st_mode | stat.S_IXUSR)
    return str(tmp_path)


def test_clock_sampler_median_and_reasons(tmp_path, monkeypatch):
    lines = [
        "0, 1500, 2070, 1350.00, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1450, 2070, 1398.10, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1520, 2070, 1301.55, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 1300, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, lines) + os.pathsep + os.environ["PATH"])
    s = bench.ClockSampler("GPU-test")
    time.sleep(0.5)
    c = s.stop()
    assert c == {"sm_mhz": 1500.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_sampler_reports_slowdowns(tmp_path, monkeypatch):
    lines = ["0, 1200, 2070, 900, 0x8, Active, Not Active, Active, Not Active"]
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, lines) + os.pathsep + os.environ["PATH"])
    s = bench.ClockSampler()
    time.sleep(0.5)
    c = s.stop()
    assert c["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"] and c["sm_mhz"] == 1200.0


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    import tempfile
    empty = tmp_path / "bin"
    empty.mkdir()
    scratch = tmp_path / "scratch"
    scratch.mkdir()
    monkeypatch.setenv("PATH", str(empty))
    monkeypatch.setattr(tempfile, "tempdir", str(scratch))
    s = bench.ClockSampler()
    assert not os.listdir(scratch)          # nothing left behind when the sampler cannot start
    assert s.stop() is None


def test_clock_sampler_removes_its_file(tmp_path, monkeypatch):
    import tempfile
    scratch = tmp_path / "scratch"
    scratch.mkdir()
    lines = ["0, 1400, 2070, 1300, 0x0, Not Active, Not Active, Not Active, Not Active"]
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, lines) + os.pathsep + os.environ["PATH"])
    monkeypatch.setattr(tempfile, "tempdir", str(scratch))
    s = bench.ClockSampler()
    time.sleep(0.3)
    assert s.stop()["sm_mhz"] == 1400.0
    assert not os.listdir(scratch)


def test_peaks_come_from_the_measured_file_or_the_fallback(tmp_path, monkeypatch):
    pk, kind = bench.peaks()
    assert kind in ("measured", "fallback")
    assert pk["bf16_tflops"] > 0 and pk["hbm_gbs"] > 0
    if kind == "measured":
        d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        assert pk["bf16_tflops"] == d["bf16_tflops"] and pk["hbm_gbs"] == d["hbm_gbs"]


def test_workload_description():
    import synth
    cfg = synth.make_config("llama-3.1-8b-20k")
    d = bench.cfg_dict(cfg, {"n_valid": 1})
    assert d["workload"] == "llama-3.1-8b-20k" and d["N"] == 160000 and d["V"] == 128256
    assert d["parallelism"] == "replicas" and d["n_valid"] == 1


def test_traffic_lookup_takes_the_committed_median_only_for_the_current_source(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    entry = {"kernel": "grpo_fwd_pair_kernel", "dram_bytes_per_launch_full_workload": 7,
             "captures": [6, 7, 9], "spread": [6, 9]}
    doc = {"kernel_source_hash": bench.kernel_source_hash(), "chunk_rows": 4864, "kernels": {"fwd": entry}}
    (prof / "traffic.json").write_text(json.dumps(doc))
    src = os.path.join(ROOT, "rl_fine_tuning_gb300")
    os.symlink(src, tmp_path / "rl_fine_tuning_gb300")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("fwd", 4864) == 7
    assert bench.ncu_traffic("fwd", 4864, "spread") == [6, 9]
    assert bench.ncu_traffic("fwd", 9728) is None          # another chunk height
    assert bench.ncu_traffic("dh", 4864) is None           # not captured
    doc["kernel_source_hash"] = "0" * 16                    # counters of another kernel source
    (prof / "traffic.json").write_text(json.dumps(doc))
    assert bench.ncu_traffic("fwd", 4864) is None
