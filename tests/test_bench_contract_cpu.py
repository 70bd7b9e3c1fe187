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


def _pairs_brute(S, W):
    return sum(min(p + 1, W) if W else p + 1 for p in range(S))


def test_accounting_matches_brute_force_and_the_stated_workload_figures():
    # visible pairs against a per-row count
    for S, W in ((1, 0), (7, 3), (129, 128), (128, 128), (300, 1), (50, 0)):
        assert bench.prefill_pairs(S, W) == _pairs_brute(S, W), (S, W)
    # the workload figures the measurements are quoted on
    assert bench.prefill_pairs(32768, 128) == 4_186_176
    assert bench.prefill_pairs(32768, 0) == 536_887_296
    assert bench.prefill_flops(32768, 64, 128) == pytest.approx(1.7147e11, rel=1e-4)
    assert bench.prefill_flops(32768, 64, 0) == pytest.approx(2.1991e13, rel=1e-4)
    assert bench.prefill_bytes(32768, 64, 8) == pytest.approx(1.5183e9, rel=1e-4)
    assert bench.prefill_bytes(32768, 64, 4) == pytest.approx(1.4345e9, rel=1e-4)
    # decode: the window ring's 131 keys per sequence at T = 4, W = 128
    lens = [9000, 131, 70000]
    assert bench.decode_pairs(lens, 4, 128) == sum(
        min(L - 4 + t + 1, 128) for L in lens for t in range(4))
    kv = sum(min(L, 131) for L in lens) * 8 * (192 + 128) * 2
    assert bench.decode_bytes(lens, 4, 64, 8, 128) == kv + 3 * 4 * 64 * (384 + 256 + 4) + 64 * 4
    # the backward's minimal products: S, dP, dV, dQ, dK
    assert bench.BWD_PAIR_FLOPS == 2 * (192 + 128 + 128 + 192 + 192)


def test_recorded_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    """roofline.traffic is reported only while the kernel's sources match
    the digest stored with the capture; otherwise null with the reason."""
    import json
    rec = {"prefill_swa_32k": {"kind": "prefill", "sources": bench.sources_digest("prefill"),
                               "dram_bytes": 123, "profile": "profiles/x.md"},
           "prefill_ga_32k": {"kind": "prefill", "sources": "0" * 16, "dram_bytes": 456,
                              "profile": "profiles/y.md"}}
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("prefill_swa_32k") == (123, "profiles/x.md")
    assert bench.recorded_traffic("prefill_ga_32k") == (None, "kernel changed since the capture")
    assert bench.recorded_traffic("decode_ga") == (None, "no capture recorded")

