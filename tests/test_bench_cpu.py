"""bench.py's reference arm on the CPU: the fp64 oracle timed on a bounded sample
of the workload, printed as one JSON line with the same metric and unit as the
CUDA arm, a cpu_baseline describing the sample, and an end-to-end figure that
moves no bytes between host and device."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_complete_line(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    assert bench.main(["--impl", "reference", "--config", "tiny_tp2_f32", "--steps", "2", "--warmup", "1"]) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["dtype"] == "f64" and d["data"] == "synthetic"
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == pytest.approx(d["value"])
    assert cb["unit"] == d["unit"] and cb["cores"] >= 1 and "tokens" in cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == pytest.approx(d["value"]) and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_attention_reference_arm_uses_the_attention_metric(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    argv = ["--impl", "reference", "--block", "attention", "--config", "attn_tiny_tp2_bf16", "--steps", "1",
            "--warmup", "0"]
    assert bench.main(argv) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.ATTN_METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["config"]["name"] == "attn_tiny_tp2_bf16"
    assert d["config"]["flops_per_step"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and "sequence" in d["cpu_baseline"]["sample"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_peak_follows_the_length_of_the_timed_region():
    """A region under a second is timed at burst clocks (burst cuBLAS peak);
    a longer one settles at the power cap (sustained peak)."""
    sys.path.insert(0, ROOT)
    import bench

    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    assert bench.choose_peak(peaks, 0.092) == (1900.0, "burst", "bf16_tflops")
    assert bench.choose_peak(peaks, 1.38) == (1700.0, "sustained", "bf16_tflops_sustained")
    assert bench.choose_peak({}, 0.5)[0] == bench.FALLBACK_PEAKS["bf16_tflops"]


def test_e2e_step_is_never_reported_below_the_device_only_step():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.e2e_guard(4.588, 4.70) == (4.70, None)
    ms, flag = bench.e2e_guard(4.588, 4.499)
    assert ms == 4.588 and "4.4990" in flag and "4.5880" in flag


def test_clock_record_keeps_only_loaded_samples():
    """Idle samples sit near the maximum clock; they must not count as under load."""
    sys.path.insert(0, ROOT)
    import bench

    def row(t, util, mhz, cap="Not Active", thermal="Not Active"):
        return {"t": t, "utilization.gpu": str(util), "clocks.sm": str(mhz), "clocks.max.sm": "2070",
                "power.draw": "900" if util else "200", "clocks_event_reasons.sw_power_cap": cap,
                "clocks_event_reasons.hw_slowdown": "Not Active",
                "clocks_event_reasons.hw_thermal_slowdown": "Not Active",
                "clocks_event_reasons.sw_thermal_slowdown": thermal}

    rows = [row(0.0, 0, 1987), row(1.0, 100, 1700, cap="Active"), row(2.0, 100, 1750), row(3.0, 100, 1800),
            row(4.0, 0, 1987, thermal="Active")]
    c = bench.summarize_clocks(rows, windows=[(1.5, 3.5)])
    assert c["samples"] == 5 and c["samples_loaded"] == 3
    assert c["sm_mhz"] == 1750 and c["sm_max_mhz"] == 2070
    assert c["samples_in_timed_regions"] == 2 and c["sm_mhz_timed_regions"] == 1775
    assert c["reasons"] == ["sw_power_cap"]  # the idle sample's reason is not a loaded one
    assert bench.parse_smi_time("2026/12/03 05:29:28.250") % 1 == 0.25
