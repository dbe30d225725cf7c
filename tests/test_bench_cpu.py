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
