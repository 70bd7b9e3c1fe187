"""The N > 1 host path of bench.py on CPU: two gloo ranks (127.0.0.1) take the
barrier, agree on the slowest rank's time and form the whole-job value; the
reference arm runs on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier(world)
        ms = 10.0 + 5.0 * rank           # rank 1 is the slow one
        m = bench.max_over_ranks(ms, world)
        value = bench.whole_job_tflops(2.0e12, world, m)
        bench.barrier(world)
        out[rank] = (m, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank, args=(world, port, out), nprocs=world, start_method="spawn",
                           join=True)
        res = dict(out)
    assert res[0] == res[1]
    m, value = res[0]
    assert m == 15.0
    # 2 ranks x 2e12 FLOPs per step in 15 ms
    assert value == pytest.approx(2 * 2.0e12 / 0.015 / 1e12)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                       text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_gpus_flag_launches_that_many_ranks():
    """`bench.py --gpus 2` started without a launcher starts two ranks itself
    (gloo here, where there is no GPU); rank 0 alone prints the line, which
    reports both ranks."""
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                        "--launch-check"], env=env, capture_output=True, text=True, timeout=300,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    import json
    out = json.loads(lines[0])
    assert out["n_gpus"] == 2 and out["max_rank"] == 1 and out["launch_check"]


def test_recorded_traffic_is_dropped_once_the_kernel_changes(tmp_path, monkeypatch):
    """The roofline's traffic figure is a recorded ncu count; it is reported
    only while the digest of the kernel's sources matches the capture's."""
    import json
    import bench
    rec = {"k": {"kind": "prefill", "sources": bench.sources_digest("prefill"),
                 "dram_bytes": 123, "profile": "profiles/x.md"}}
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("k") == (123, "profiles/x.md")
    rec["k"]["sources"] = "0" * 16
    f.write_text(json.dumps(rec))
    assert bench.recorded_traffic("k")[0] is None
    assert bench.recorded_traffic("missing")[0] is None
