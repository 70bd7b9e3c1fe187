"""bench.py's reference arm (the fp64 oracle on the host cores) prints the
contract's line: checked on CPU with the two prefill workloads shrunk so the
run takes seconds (the arithmetic is the oracle's either way)."""
import argparse
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


@pytest.fixture
def small_workloads(monkeypatch):
    cfg = dict(synth.CONFIGS)
    cfg["swa_prefill_32k"] = dict(cfg["swa_prefill_32k"], seqlens=[512], hq=8, hkv=1)
    cfg["ga_prefill_32k"] = dict(cfg["ga_prefill_32k"], seqlens=[256], hq=8, hkv=2)
    monkeypatch.setattr(synth, "CONFIGS", cfg)
    monkeypatch.setattr(bench, "_CPU_CASES", {})


def test_reference_line_has_the_contract_keys(small_workloads):
    args = argparse.Namespace(steps=2, warmup=1, cpu_budget=0.5)
    out = bench.run_reference(args)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert k in out, k
    assert out["impl"] == "reference" and out["steps"] == 2 and out["warmup"] == 1
    assert out["value"] > 0 and out["unit"] == "TFLOP/s" and out["dtype"] == "f64"
    cb = out["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == out["value"] and cb["cores"] >= 1
    assert "rows" in cb["sample"]
    e = out["e2e"]
    assert e["value"] == out["value"] and e["unit"] == out["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_whole_job_value_is_weak_scaling():
    assert bench.whole_job_tflops(1e12, 1, 1000.0) == pytest.approx(1.0)
    assert bench.whole_job_tflops(1e12, 4, 1000.0) == pytest.approx(4.0)
