"""Host logic of bench.py (no GPU): the clock record, the DRAM-traffic gate, the kernel the bench
reports for W1/W2, and the reference arm's JSON line on a small workload."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as wl  # noqa: E402

SMI = "0, %d, 2032, 900.00, %d, 0x4, Not Active, Not Active, Not Active, %s"


def _sampler(nvml, smi_lines, region):
    c = bench.ClockSampler(0)
    c.nvml = list(nvml)
    c.nvml_max = 2032.0
    c.lines = list(smi_lines)
    c.region = list(region)
    return c


def test_clock_summary_takes_the_nvml_samples_inside_the_timed_region():
    nvml = [(0.0, 2032.0, 0x0), (1.0, 1500.0, 0x4), (1.1, 1600.0, 0x4), (1.2, 1700.0, 0x0), (5.0, 2032.0, 0x0)]
    c = _sampler(nvml, [SMI % (2032, 100, "Active")], (0.5, 2.0))
    s = c.summary()
    assert s["source"].startswith("NVML")
    assert s["samples"] == 3 and s["sm_mhz"] == 1600.0 and s["sm_mhz_min"] == 1500.0
    assert s["reasons"] == ["sw_power_cap"]
    assert s["nvidia_smi"]["samples"] == 1


def test_clock_summary_reports_slowdown_reasons():
    nvml = [(1.0, 1200.0, 0x8), (1.1, 1200.0, 0x40), (1.2, 1200.0, 0x20 | 0x4)]
    s = _sampler(nvml, [], (0.0, 2.0)).summary()
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap", "sw_thermal_slowdown"]


def test_clock_summary_falls_back_to_nvidia_smi():
    lines = [SMI % (1980, 95, "Active"), SMI % (2032, 10, "Not Active"), SMI % (1900, 90, "Not Active")]
    s = _sampler([(1.0, 1500.0, 0x4)], lines, (0.0, 2.0)).summary()   # one NVML sample: too few
    assert s["source"].startswith("nvidia-smi")
    assert s["sm_mhz"] == (1980 + 1900) / 2 and s["samples_under_load"] == 2
    assert s["reasons"] == ["sw_power_cap"]
    assert _sampler([], [], (0.0, 1.0)).summary() is None


def test_traffic_is_reported_only_for_the_captured_source(monkeypatch):
    assert bench.traffic_for("mixtral_prefill") == bench.NCU_TRAFFIC["bytes_per_launch"]["mixtral_prefill"]
    monkeypatch.setitem(bench.NCU_TRAFFIC, "code_sha256", "0" * 64)
    assert bench.traffic_for("mixtral_prefill") is None


def test_source_hash_ignores_comments(tmp_path):
    a, b, c = tmp_path / "a.cu", tmp_path / "b.cu", tmp_path / "c.cu"
    a.write_text("int f() {\n  return 1;  // one\n}\n")
    b.write_text("// header\nint f() {\n\n  return 1;\n}\n")
    c.write_text("int f() {\n  return 2;\n}\n")
    assert bench._code_sha256(str(a)) == bench._code_sha256(str(b)) != bench._code_sha256(str(c))


def test_reported_w12_kernel(monkeypatch):
    monkeypatch.delenv("MOE_GEMM_KERNEL", raising=False)
    W = wl.WORKLOADS
    assert [bench.gemm_variant(W[n]) for n in ("mixtral_prefill", "hunyuan_a13b", "deepseek_v3")] == ["tpairw"] * 3
    assert bench.gemm_variant(W["mixtral_decode"]) == "single"
    assert bench.gemm_variant(W["tiny_f32"]) == "simt"
    monkeypatch.setenv("MOE_GEMM_KERNEL", "pair")
    assert bench.gemm_variant(W["mixtral_prefill"]) == "pair"


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_f32", "--steps", "2", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3
    assert line["unit"] == "tokens/s" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["config"]["workload"] == "tiny_f32"
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == line["value"] and cpu["cores"] >= 1 and cpu["sample"]
