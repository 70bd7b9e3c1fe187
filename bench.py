"""Benchmark of the hybrid SWA / GA sink-attention hot path on B300.

One step = one pass of the whole path over one batch of synthetic inputs:
  1. SWA layer prefill, seq 32768, 64 query / 8 KV heads, W = 128, base 1e4
  2. GA layer prefill, seq 32768, 64 query / 4 KV heads, global, base 5e6
  3. decode / MTP-verify of one hybrid block, batch 64 x 4 query tokens:
     append of the 4 new tokens + decode, for its five SWA layers (each a
     131-slot ring, 8 KV heads; called back to back) and its GA layer
     (lengths uniform in [8K, 64K], 4 KV heads)
All inputs are bf16 ~ N(0, 1), sinks ~ N(0, 1) (seeded, synthetic).

Prints ONE JSON line (rank 0).  `value` = algorithmic FLOPs of the step /
device time of the step (TFLOP/s); per-part TFLOP/s, GB/s and roofline
fractions are in `parts`; `roofline` covers the dominant kernel (GA prefill).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl cuda|reference]

With --impl reference the CPU oracle is timed instead, on bounded row samples
of the same workload (the rows of attention are independent, so a sample of
rows is an exact sample of the work).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "prefill TFLOP/s & decode HBM GB/s (SWA+GA sink attention) vs B300 roofline"
D_QK, D_V, R = 192, 128, 64
DECODE_SWA_LAYERS = 5  # window layers per hybrid block (5 SWA : 1 GA)
PAIR_FLOPS = 2 * (D_QK + D_V)  # FLOPs per (query row, visible key) pair and head


# --------------------------------------------------------------------- accounting
def prefill_pairs(S: int, W: int) -> int:
    """Visible (query, key) pairs of one head of one sequence."""
    if W == 0 or W >= S:
        return S * (S + 1) // 2
    return W * (W + 1) // 2 + (S - W) * W


def prefill_flops(S, hq, W):
    return PAIR_FLOPS * hq * prefill_pairs(S, W)


def prefill_bytes(S, hq, hkv):
    # q, k, v read once, sink read once, out (bf16) and lse (fp32) written once
    return S * (hq * D_QK * 2 + hkv * D_QK * 2 + hkv * D_V * 2 + hq * D_V * 2 + hq * 4) + hq * 4


def decode_pairs(lens, T, W):
    tot = 0
    for L in lens:
        for t in range(T):
            p = L - T + t
            tot += min(p + 1, W) if W else p + 1
    return tot


def decode_bytes(lens, T, hq, hkv, W):
    keys = sum(min(L, W + T - 1) if W else L for L in lens)
    kv = keys * hkv * (D_QK + D_V) * 2
    qo = len(lens) * T * hq * (D_QK * 2 + D_V * 2 + 4)
    return kv + qo + hq * 4


def append_bytes(B, T, hkv):
    return B * T * hkv * (D_QK + D_V) * 2 * 2 + B * 4  # read new k/v, write cache slots


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # the timed region starts once sampling has (up to 3 s)
            t_end = time.time() + 3.0
            while not self.lines and time.time() < t_end and self.proc.poll() is None:
                time.sleep(0.01)
            self.lines.clear()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def copy_note(copy_ms, alone_ms, nbytes, hbm):
    """A part against a device-to-device copy moving the same bytes: the
    copy's time and fraction of the HBM peak, and the part's time (alone)
    over the copy's."""
    return {"ms": round(copy_ms, 5), "frac_of_hbm_peak": round(nbytes / copy_ms / 1e6 / hbm, 4),
            "part_alone_over_copy": round(alone_ms / copy_ms, 3)}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"], "measured"
    except (OSError, KeyError, ValueError):
        return 6400.0, 1800.0, 1400.0, "fallback"


# Which bf16 peak a kernel's FLOP rate is divided by.  The burst figure (a
# cuBLAS GEMM timed alone, SM clock near its 2032 MHz maximum) fits a kernel
# that runs for milliseconds inside a step whose own clock record stays near
# the maximum; the sustained figure (the same GEMM back to back for seconds,
# SM clock pulled down by the power cap) fits a kernel that itself runs for
# seconds.  The line records which one each fraction used.
SUSTAINED_AFTER_S = 1.0


def tensor_peak(kernel_s, tf_burst, tf_sust):
    if kernel_s >= SUSTAINED_AFTER_S:
        return tf_sust, "bf16_tflops_sustained"
    return tf_burst, "bf16_tflops"


# DRAM traffic per launch of a kernel, as counted by one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), with a digest of the sources
# the kernel was built from: once the sources change, the count no longer
# describes the kernel and the line reports null.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = {
    "prefill": ["prefill_tc.cu", "rope_append.cu", "common.cuh", "hattn_internal.h"],
    "decode": ["decode.cu", "rope_append.cu", "common.cuh", "hattn_internal.h"],
    "backward": ["backward.cu", "common.cuh", "hattn_internal.h"],
}


def sources_digest(kind):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "global_attention_sinks_gqa_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(key):
    """(bytes per launch, source note) of a recorded capture, or (None, why)."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)[key]
    except (OSError, KeyError, ValueError):
        return None, "no capture recorded"
    if rec.get("sources") != sources_digest(rec["kind"]):
        return None, "kernel changed since the capture"
    return rec["dram_bytes"], rec["profile"]


def step_config(world: int = 1):
    return {"workload": "swa_prefill_32k + ga_prefill_32k + decode_b64_t4 (5 x swa ring 131 "
                        "+ ga 8K-64K)",
            "swa_prefill": "seq 32768, 64q/8kv, W=128, d_qk 192, d_v 128, rope 64 @1e4",
            "ga_prefill": "seq 32768, 64q/4kv, global, rope 64 @5e6",
            "decode": "batch 64 x 4 verify tokens; 5 swa layers (8kv ring 131 each) + 1 ga "
                      "layer (4kv, L~U[8192,65536])",
            "l2": "inputs larger than L2 (no flush needed); parts' alone_ms: each part's "
                  "calls repeated on their own, L2 flushed between repetitions",
            "parallelism": f"replicas x{world}"}


# --------------------------------------------------------------------- CUDA arm
class Workload:
    """Device-resident inputs and outputs of one step, plus pinned host copies
    of the per-step inputs for the end-to-end measurement."""

    def __init__(self, dev):
        import global_attention_sinks_gqa_b300 as ha
        self.ha = ha
        self.dev = dev
        cf = synth.CONFIGS
        self.layers = []
        for name in ("swa_prefill_32k", "ga_prefill_32k"):
            c = cf[name]
            pc = synth.prefill_case(c["seqlens"], c["hq"], c["hkv"], window=c["window"],
                                    rope_base=c["rope_base"], seed=c["seed"], device=dev)
            S = pc.total
            lay = dict(name=name, case=pc, S=S,
                       out=torch.empty((S, pc.hq, D_V), dtype=torch.bfloat16, device=dev),
                       lse=torch.empty((S, pc.hq), dtype=torch.float32, device=dev),
                       ws=torch.empty(ha.hattn_prefill_workspace_size(S, pc.hkv, D_QK),
                                      dtype=torch.uint8, device=dev),
                       flops=prefill_flops(S, pc.hq, pc.window),
                       bytes=prefill_bytes(S, pc.hq, pc.hkv))
            self.layers.append(lay)
        dc = cf["decode_b64_t4"]
        self.B, self.T = dc["B"], dc["T"]
        self.lens = synth.random_lengths(self.B, dc["lens"][0], dc["lens"][1], dc["seed"])
        self.lmax = dc["lens"][1]
        # the decode step of one hybrid block: its five window layers (each
        # with its own 131-slot ring), called back to back, then its global layer
        self.dec = []
        for kind, cap, ring, nl in (("swa", 131, True, DECODE_SWA_LAYERS),
                                    ("ga", self.lmax, False, 1)):
            p = dc[kind]
            for li in range(nl):
                dd = self._decode_layer(p, cap, ring, dc["seed"] + (0 if ring else 1) + 100 * li)
                dd.update(kind=kind, cap=cap, ring=ring, p=p, layer=li)
                self.dec.append(dd)

    def _decode_layer(self, p, cap, ring, seed):
        ha, dev, B, T = self.ha, self.dev, self.B, self.T
        hq, hkv = p["hq"], p["hkv"]
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        kc = torch.empty((B, hkv, cap, D_QK), dtype=torch.bfloat16, device=dev)
        vc = torch.empty((B, hkv, cap, D_V), dtype=torch.bfloat16, device=dev)
        # history before the step: written by the append kernel, chunk by chunk
        chunk = 4096 if not ring else cap
        for b, L in enumerate(self.lens):
            hist = L - T
            s0 = max(0, hist - cap) if ring else 0
            for s in range(s0, hist, chunk):
                n = min(chunk, hist - s)
                k = synth.randn_bf16((1, n, hkv, D_QK), g, dev)
                v = synth.randn_bf16((1, n, hkv, D_V), g, dev)
                ha.rope_kv_append(k, v, torch.tensor([s], dtype=torch.int32, device=dev),
                                  kc[b:b + 1], vc[b:b + 1], is_ring=ring,
                                  rope_base=p["rope_base"])
        q = synth.randn_bf16((B, T, hq, D_QK), g, dev)
        k_new = synth.randn_bf16((B, T, hkv, D_QK), g, dev)
        v_new = synth.randn_bf16((B, T, hkv, D_V), g, dev)
        sink = synth.randn_f32((hq,), g, dev)
        sl = torch.tensor(self.lens, dtype=torch.int32, device=dev)
        ws_n = ha.hattn_decode_workspace_size(B, T, hq, hkv, D_V, self.lmax, p["window"], cap,
                                              1 if ring else 0)
        ws = torch.empty(max(ws_n, 256), dtype=torch.uint8, device=dev)
        return dict(q=q, k_new=k_new, v_new=v_new, sink=sink, kc=kc, vc=vc, seqlens=sl,
                    start=sl - T, ws=ws, ws_n=ws_n,
                    out=torch.empty((B, T, hq, D_V), dtype=torch.bfloat16, device=dev),
                    lse=torch.empty((B, T, hq), dtype=torch.float32, device=dev),
                    flops=PAIR_FLOPS * hq * decode_pairs(self.lens, T, p["window"]),
                    bytes=decode_bytes(self.lens, T, hq, hkv, p["window"]),
                    abytes=append_bytes(B, T, hkv))

    # one C-ABI call per hot-path step; returns number of kernel launches
    def run_prefill(self, lay, stream, q=None, k=None, v=None):
        ha, c = self.ha, lay["case"]
        st = ha.hattn_prefill(c.q if q is None else q, c.k if k is None else k,
                              c.v if v is None else v, c.sink, lay["out"], lay["lse"], 1,
                              c.cu_seqlens, lay["S"], lay["S"], c.hq, c.hkv, D_QK, D_V, R,
                              c.rope_base, c.window, c.scale, lay["ws"], lay["ws"].numel(),
                              stream)
        assert st == 0, ha.status_string(st)
        return 2

    def run_decode(self, dd, stream, q=None, k_new=None, v_new=None):
        """One decode / verify step of the layer: the append of the T new
        tokens and the attention over the cache, one C-ABI call."""
        ha, p = self.ha, dd["p"]
        st = ha.hattn_decode_append(dd["q"] if q is None else q,
                                    dd["k_new"] if k_new is None else k_new,
                                    dd["v_new"] if v_new is None else v_new, dd["kc"], dd["vc"],
                                    dd["seqlens"], dd["sink"], dd["out"], dd["lse"], self.B,
                                    self.T, p["hq"], p["hkv"], D_QK, D_V, dd["cap"],
                                    1 if dd["ring"] else 0, p["window"], self.lmax, R,
                                    p["rope_base"], 1.0 / math.sqrt(D_QK), dd["ws"],
                                    dd["ws"].numel(), stream)
        assert st == 0, ha.status_string(st)
        # a ring of <= 144 slots with <= 32 rows per KV head runs the append
        # inside the attention kernel; otherwise the append kernel goes first
        fused = (dd["ring"] and dd["cap"] <= 144 and self.T <= 4
                 and (p["hq"] // p["hkv"]) * self.T <= 32)
        return (1 if fused else 2) + (1 if dd["ws_n"] else 0)

    def flops(self):
        return sum(l["flops"] for l in self.layers) + sum(d["flops"] for d in self.dec)


def run_cuda(args, rank, world):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl = Workload(dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    torch.cuda.synchronize()

    def step(events=None):
        n = 0
        for i, lay in enumerate(wl.layers):
            if events is not None:
                events[f"p{i}"][0].record(stream)
            n += wl.run_prefill(lay, sptr)
            if events is not None:
                events[f"p{i}"][1].record(stream)
        # the window layers' calls back to back (one event pair around them),
        # then the global layer's
        for kind in ("swa", "ga"):
            if events is not None:
                events[f"d_{kind}"][0].record(stream)
            for dd in wl.dec:
                if dd["kind"] == kind:
                    n += wl.run_decode(dd, sptr)
            if events is not None:
                events[f"d_{kind}"][1].record(stream)
        return n

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    wl.ha.check_device_status()
    keys = ["p0", "p1", "d_swa", "d_ga"]
    ev = [{k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for k in keys} for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        torch.cuda.nvtx.range_push("timed")
        start.record(stream)
        for s in range(args.steps):
            launches += step(ev[s])
        stop.record(stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    barrier(world)
    total_ms = start.elapsed_time(stop)
    ms = max_over_ranks(total_ms, world) / args.steps
    part_ms = {k: statistics.mean(e[k][0].elapsed_time(e[k][1]) for e in ev) for k in keys}
    wl.ha.check_device_status()

    # Each part alone as well (its calls back to back, same inputs), outside
    # the step: inside the step every part runs under the SM clock the
    # power-capped global prefill leaves behind; alone, the short parts run
    # at their own clock.  The step's numbers above stay the reported ones.
    # The flush (8 times the L2) also gives the host ~160 us to enqueue the
    # part's calls before the GPU reaches the start event, so that the
    # Python marshalling of short parts (five decode calls) is not timed.
    flush = torch.empty(1 << 30, dtype=torch.uint8, device=dev)

    def alone(fn, reps):
        fn()
        ev_a = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(reps)]
        for a0, a1 in ev_a:
            flush.zero_()  # L2 flushed between repetitions, outside the timed calls
            a0.record(stream)
            fn()
            a1.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a0.elapsed_time(a1) for a0, a1 in ev_a)

    alone_ms = {
        "p0": alone(lambda: wl.run_prefill(wl.layers[0], sptr), 20),
        "d_swa": alone(lambda: [wl.run_decode(dd, sptr) for dd in wl.dec if dd["kind"] == "swa"],
                       20),
        "d_ga": alone(lambda: [wl.run_decode(dd, sptr) for dd in wl.dec if dd["kind"] == "ga"],
                      10),
    }
    wl.ha.check_device_status()

    # The HBM peak is a device-to-device copy of 2 GiB each way; at the size
    # of a short HBM-bound part the same copy reaches much less of it (ramp
    # and tail).  So the HBM-bound parts also get a copy moving their own
    # bytes (half read, half written), chained like their calls (the window
    # decode: five layers, five buffers), L2 flushed before each repetition.
    def copy_of(nbytes, chain):
        n = int(nbytes) // 2 // 16 * 16  # bytes each way
        src = [torch.zeros(n, dtype=torch.uint8, device=dev) for _ in range(chain)]
        dst = [torch.empty(n, dtype=torch.uint8, device=dev) for _ in range(chain)]
        t = alone(lambda: [d.copy_(x) for x, d in zip(src, dst)], 20)
        del src, dst
        return t / chain

    swa_dec = [dd for dd in wl.dec if dd["kind"] == "swa"]
    copy_ms = {"p0": copy_of(wl.layers[0]["bytes"], 1),
               "d_swa": copy_of(swa_dec[0]["bytes"] + swa_dec[0]["abytes"], len(swa_dec))}

    # ---- end to end: per step, inputs from pinned host memory, outputs back
    e2e = run_e2e(wl, args, stream, sptr)

    hbm, tf_burst, tf_sust, src = measured_peaks()
    clocks = clk.summary()
    parts = {}
    for i, lay in enumerate(wl.layers):
        t = part_ms[f"p{i}"] / 1e3
        tf, tf_name = tensor_peak(t, tf_burst, tf_sust)
        bound_f = lay["flops"] / (tf * 1e12)
        bound_b = lay["bytes"] / (hbm * 1e9)
        parts[lay["name"]] = dict(ms=part_ms[f"p{i}"], tflops=lay["flops"] / t / 1e12,
                                  gbs=lay["bytes"] / t / 1e9,
                                  roofline_frac=max(bound_f, bound_b) / t,
                                  bound="tensor" if bound_f > bound_b else "hbm",
                                  peak="hbm_gbs" if bound_b > bound_f else tf_name)
        if f"p{i}" in alone_ms:
            ta = alone_ms[f"p{i}"] / 1e3
            parts[lay["name"]].update(alone_ms=ta * 1e3,
                                      alone_roofline_frac=max(bound_f, bound_b) / ta)
        if f"p{i}" in copy_ms:
            parts[lay["name"]]["same_bytes_copy"] = copy_note(
                copy_ms[f"p{i}"], alone_ms[f"p{i}"], lay["bytes"], hbm)
        tr, _ = recorded_traffic("prefill_" + lay["name"].split("_")[0] + "_32k")
        parts[lay["name"]]["traffic"] = tr
    for kind in ("swa", "ga"):
        lays = [dd for dd in wl.dec if dd["kind"] == kind]
        t = part_ms[f"d_{kind}"] / 1e3 / len(lays)  # per layer
        dd = lays[0]
        byts = dd["bytes"] + dd["abytes"]
        parts[f"decode_{kind}_b64_t4"] = dict(
            ms=t * 1e3, tflops=dd["flops"] / t / 1e12, gbs=byts / t / 1e9,
            roofline_frac=byts / (hbm * 1e9) / t, bound="hbm", peak="hbm_gbs",
            verify_tokens_per_s=wl.B * wl.T / t, layers=len(lays),
            timing="per layer: one event pair around the layers' calls back to back",
            alone_ms=alone_ms[f"d_{kind}"] / len(lays),
            alone_roofline_frac=byts / (hbm * 1e9) / (alone_ms[f"d_{kind}"] / len(lays) / 1e3))
        if f"d_{kind}" in copy_ms:
            parts[f"decode_{kind}_b64_t4"]["same_bytes_copy"] = copy_note(
                copy_ms[f"d_{kind}"], alone_ms[f"d_{kind}"] / len(lays), byts, hbm)
    ga = wl.layers[1]
    ga_s = part_ms["p1"] / 1e3
    ga_tf, ga_tf_name = tensor_peak(ga_s, tf_burst, tf_sust)
    ga_traffic, ga_traffic_src = recorded_traffic("prefill_ga_32k")
    flops = wl.flops()
    value = whole_job_tflops(flops, world, ms)
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q/k/v, N(0,1) fp32 sinks)",
        "config": step_config(world),
        "parts": parts,
        "roofline": {"bound": "tensor", "kernel": "prefill GA (hattn_prefill window=0: "
                                                  "key-rotation pass + prefill_kernel)",
                     "achieved": round(ga["flops"] / ga_s / 1e12, 2),
                     "peak": ga_tf, "unit": "TFLOP/s",
                     "frac": round(ga["flops"] / ga_s / 1e12 / ga_tf, 4),
                     "traffic": ga_traffic, "traffic_source": ga_traffic_src,
                     "algorithmic_bytes": ga["bytes"],
                     "peak_source": f"{src} {ga_tf_name} (of measured; step SM clock median "
                                    f"{clocks.get('sm_mhz')} MHz)"},
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if args.extras and world == 1:
        # the other workloads of the path, timed after the step on the same
        # GPU: the hybrid block at 256K (a10) and the backward of both layers
        del wl
        torch.cuda.empty_cache()
        out["extra_workloads"] = {
            "hybrid_block_256k": _extra(run_hybrid_block(argparse.Namespace(steps=2, warmup=1))),
            "backward_32k": _extra(run_backward(argparse.Namespace(steps=5, warmup=3))),
        }
    if rank == 0 and args.cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_budget)
    return out


def _extra(line):
    """A workload's own result line, less the keys the main line already states."""
    drop = ("metric", "data", "higher_is_better", "scaling", "vs_baseline", "dtype", "n_gpus")
    return {k: v for k, v in line.items() if k not in drop}


def run_e2e(wl, args, stream, sptr):
    """Same step through the C ABI with host-resident inputs: each step copies
    its inputs (q, k, v of both prefill layers; q and the new k/v of both decode
    layers) from pinned host memory and reads the outputs back."""
    dev = wl.dev
    host_in, dev_in = [], []
    for lay in wl.layers:
        c = lay["case"]
        hs = [t.cpu().pin_memory() for t in (c.q, c.k, c.v)]
        host_in.append(hs)
        dev_in.append([torch.empty_like(t, device=dev) for t in hs])
    for dd in wl.dec:
        hs = [t.cpu().pin_memory() for t in (dd["q"], dd["k_new"], dd["v_new"])]
        host_in.append(hs)
        dev_in.append([torch.empty_like(t, device=dev) for t in hs])
    outs = [l["out"] for l in wl.layers] + [d["out"] for d in wl.dec]
    lses = [l["lse"] for l in wl.layers] + [d["lse"] for d in wl.dec]
    host_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    host_lse = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in lses]
    h2d = sum(t.numel() * t.element_size() for hs in host_in for t in hs)
    d2h = sum(t.numel() * t.element_size() for t in host_out + host_lse)

    # Copies overlap the layers: uploads run on one copy stream, read-backs on
    # another, the C-ABI calls on the compute stream.  Part i's inputs go up
    # as soon as the previous step's part i no longer needs its buffers (so
    # the next step's uploads run under this step's layers), and its outputs
    # come back while the next part computes; part i's next call waits for
    # that read-back before rewriting its outputs.
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    nparts = len(dev_in)
    uploaded = [torch.cuda.Event() for _ in range(nparts)]
    computed = [torch.cuda.Event() for _ in range(nparts)]
    read_back = [torch.cuda.Event() for _ in range(nparts)]
    part_outs = [[outs[i], lses[i]] for i in range(nparts)]
    part_host = [[host_out[i], host_lse[i]] for i in range(nparts)]

    def run_part(i):
        if i < len(wl.layers):
            wl.run_prefill(wl.layers[i], sptr, *dev_in[i])
        else:
            wl.run_decode(wl.dec[i - len(wl.layers)], sptr, *dev_in[i])

    def step():
        for i in range(nparts):
            up.wait_event(computed[i])  # the previous step's part i is done with its inputs
            with torch.cuda.stream(up):
                for h, d in zip(host_in[i], dev_in[i]):
                    d.copy_(h, non_blocking=True)
            uploaded[i].record(up)
        for i in range(nparts):
            stream.wait_event(uploaded[i])
            stream.wait_event(read_back[i])  # the previous step's outputs of part i are home
            run_part(i)
            computed[i].record(stream)
            down.wait_event(computed[i])
            with torch.cuda.stream(down):
                for o, h in zip(part_outs[i], part_host[i]):
                    h.copy_(o, non_blocking=True)
            read_back[i].record(down)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(1, min(args.steps, 5))
    start.record(stream)
    up.wait_event(start)
    down.wait_event(start)
    for _ in range(n):
        step()
    stream.wait_stream(up)
    stream.wait_stream(down)
    stop.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(stop) / n

    # the same copies alone (no layer calls), for the floor they set
    def copies():
        with torch.cuda.stream(up):
            for i in range(nparts):
                for h, d in zip(host_in[i], dev_in[i]):
                    d.copy_(h, non_blocking=True)
        with torch.cuda.stream(down):
            for i in range(nparts):
                for o, h in zip(part_outs[i], part_host[i]):
                    h.copy_(o, non_blocking=True)

    copies()
    torch.cuda.synchronize()
    start.record(stream)
    up.wait_event(start)
    down.wait_event(start)
    for _ in range(n):
        copies()
    stream.wait_stream(up)
    stream.wait_stream(down)
    stop.record(stream)
    torch.cuda.synchronize()
    copy_ms = start.elapsed_time(stop) / n
    return {"value": round(wl.flops() / (ms / 1e3) / 1e12, 3), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 3), "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h),
            "copies": "uploads and read-backs on two copy streams, overlapping the layers",
            "copies_alone_ms": round(copy_ms, 3)}


# --------------------------------------------------------------------- CPU oracle arm
_CPU_CASES = {}


def _cpu_case(name):
    """The seeded host copy of a prefill workload (built once per process)."""
    if name not in _CPU_CASES:
        c = synth.CONFIGS[name]
        _CPU_CASES[name] = synth.prefill_case(c["seqlens"], c["hq"], c["hkv"], window=c["window"],
                                              rope_base=c["rope_base"], seed=c["seed"])
    return _CPU_CASES[name]


def cpu_baseline(budget_s: float = 20.0):
    """The fp64 oracle as it stands, timed on this host's cores on a bounded row
    sample of the same step (about budget_s seconds of CPU work: a third on
    sliding-window rows, the rest on global rows); reported as algorithmic
    TFLOP/s of the sample."""
    import oracle
    cf = synth.CONFIGS
    done_flops, secs = 0.0, 0.0
    samples = []
    # SWA prefill rows (32K, 64/8): rows are independent; evenly spaced batches
    c = cf["swa_prefill_32k"]
    pc = _cpu_case("swa_prefill_32k")
    S = pc.total
    n_rows, t0 = 0, time.perf_counter()
    rs = np.random.RandomState(0)
    while time.perf_counter() - t0 < budget_s / 3 and n_rows < S:
        rows = np.sort(rs.choice(S, size=512, replace=False))
        oracle.prefill(pc.q, pc.k, pc.v, pc.sink, [0, S], window=c["window"],
                       rope_base=c["rope_base"], scale=pc.scale, rows=rows)
        done_flops += sum(PAIR_FLOPS * pc.hq * min(int(r) + 1, c["window"]) for r in rows)
        n_rows += len(rows)
    secs += time.perf_counter() - t0
    samples.append(f"swa_prefill_32k: {n_rows} of {S} rows")
    # GA prefill rows (32K, 64/4): rows spread over the sequence until the budget is spent
    c = cf["ga_prefill_32k"]
    pc = _cpu_case("ga_prefill_32k")
    S = pc.total
    order = rs.permutation(S)
    n_ok, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s - secs and n_ok < S:
        r = int(order[n_ok])
        oracle.prefill(pc.q, pc.k, pc.v, pc.sink, [0, S], window=0, rope_base=c["rope_base"],
                       scale=pc.scale, rows=[r])
        done_flops += PAIR_FLOPS * pc.hq * (r + 1)
        n_ok += 1
    secs += time.perf_counter() - t0
    samples.append(f"ga_prefill_32k: {n_ok} random rows of {S}")
    return {"value": round(done_flops / secs / 1e12, 6), "unit": "TFLOP/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "; ".join(samples) + f"; {secs:.1f} s of fp64 CPU work"}


def run_reference(args):
    """--impl reference: the CPU oracle as the reference arm, K bounded steps."""
    import oracle
    steps_ms = []
    # each step a bounded sample: the whole run stays within a few minutes
    budget = max(2.0, min(args.cpu_budget, 120.0 / max(1, args.steps)))
    for _ in range(args.warmup):
        cpu_baseline(budget_s=1.0)
    vals = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        cb = cpu_baseline(budget_s=budget)
        steps_ms.append((time.perf_counter() - t0) * 1e3)
        vals.append(cb["value"])
    v = statistics.mean(vals)
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(statistics.mean(steps_ms), 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1))",
            "config": step_config(1),
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": cb["sample"]},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# --------------------------------------------------------------------- distributed
def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """The largest of the ranks' x (every rank gets it): the job's time is its
    slowest rank's."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def launch_replicas(n, argv):
    """Start n ranks of this script on this node (torch's launcher, rendezvous
    on 127.0.0.1), one per local GPU; rank 0 prints the line.  Returns the
    launcher's exit status."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr=127.0.0.1", f"--master-port={port}",
           os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def launch_check(rank, world):
    """The replica launch without attention work: every rank meets the others
    at a barrier and the line carries the largest rank and the world size."""
    barrier(world)
    top = max_over_ranks(float(rank), world)
    return {"launch_check": True, "n_gpus": world, "max_rank": int(top),
            "backend": __import__("torch.distributed", fromlist=["x"]).get_backend()
            if world > 1 else None}


def whole_job_tflops(flops_per_rank_step, world, ms_per_step):
    """Whole-job throughput: every rank runs the same step (weak scaling), the
    step takes the slowest rank's time."""
    return flops_per_rank_step * world / (ms_per_step / 1e3) / 1e12


def run_hybrid_block(args):
    """One hybrid block at seq 262144 -- 5 sliding-window layers (64q/8kv,
    W=128, base 1e4) then 1 global layer (64q/4kv, base 5e6), fresh N(0,1) inputs
    per layer, all resident in HBM; one step = the 6 layer calls."""
    import global_attention_sinks_gqa_b300 as ha
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    cfg = synth.CONFIGS["hybrid_block_256k"]
    S = cfg["seqlens"][0]
    layers = []
    for li in range(cfg["n_swa"] + 1):
        kind = "swa" if li < cfg["n_swa"] else "ga"
        p = cfg[kind]
        c = synth.prefill_case([S], p["hq"], p["hkv"], window=p["window"],
                               rope_base=p["rope_base"], seed=cfg["seed"] * 100 + li, device=dev)
        layers.append(dict(kind=kind, case=c,
                           out=torch.empty((S, c.hq, D_V), dtype=torch.bfloat16, device=dev),
                           lse=torch.empty((S, c.hq), dtype=torch.float32, device=dev),
                           ws=torch.empty(ha.hattn_prefill_workspace_size(S, c.hkv, D_QK),
                                          dtype=torch.uint8, device=dev),
                           flops=prefill_flops(S, c.hq, c.window),
                           bytes=prefill_bytes(S, c.hq, c.hkv)))
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream

    def step(ev=None):
        for i, lay in enumerate(layers):
            c = lay["case"]
            if ev is not None:
                ev[i][0].record(stream)
            st = ha.hattn_prefill(c.q, c.k, c.v, c.sink, lay["out"], lay["lse"], 1, c.cu_seqlens,
                                  S, S, c.hq, c.hkv, D_QK, D_V, R, c.rope_base, c.window,
                                  c.scale, lay["ws"], lay["ws"].numel(), sptr)
            assert st == 0, ha.status_string(st)
            if ev is not None:
                ev[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ha.check_device_status()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in layers] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        start.record(stream)
        for k in range(args.steps):
            step(ev[k])
        stop.record(stream)
        torch.cuda.synchronize()
    ha.check_device_status()
    ms = start.elapsed_time(stop) / args.steps
    hbm, tf_burst, tf_sust, src = measured_peaks()
    flops = sum(l["flops"] for l in layers)
    byts = sum(l["bytes"] for l in layers)
    parts = {}
    frac = 0.0
    for i, lay in enumerate(layers):
        t = statistics.mean(e[i][0].elapsed_time(e[i][1]) for e in ev) / 1e3
        tf, tf_name = tensor_peak(t, tf_burst, tf_sust)
        bf = lay["flops"] / (tf * 1e12)
        bb = lay["bytes"] / (hbm * 1e9)
        frac += max(bf, bb)
        parts[f"layer{i}_{lay['kind']}"] = dict(ms=t * 1e3, tflops=lay["flops"] / t / 1e12,
                                                 gbs=lay["bytes"] / t / 1e9,
                                                 roofline_frac=max(bf, bb) / t,
                                                 peak="hbm_gbs" if bb > bf else tf_name)
    return {"metric": METRIC, "value": round(flops / (ms / 1e3) / 1e12, 3), "unit": "TFLOP/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 q/k/v, N(0,1) fp32 sinks)",
            "config": {"workload": "hybrid_block_256k: seq 262144, 5 SWA layers (64q/8kv, W=128, "
                                   "base 1e4) + 1 GA layer (64q/4kv, base 5e6)",
                       "l2": "inputs larger than L2 (no flush needed)"},
            "block_roofline_frac": round(frac / (ms / 1e3), 4),
            "algorithmic": {"flops": flops, "bytes": byts},
            "parts": parts, "clocks": clk.summary()}


def run_prefix_prefill(args):
    """Prefill over a cached prefix: a global layer (64q/4kv, base 5e6) whose
    cache already holds 28672 tokens receives 4096 new ones (append + attention,
    one hattn_prefill_cached call per step)."""
    import global_attention_sinks_gqa_b300 as ha
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    P, S = 28672, 4096
    p = synth.CONFIGS["ga_prefill_32k"]
    hq, hkv, base = p["hq"], p["hkv"], p["rope_base"]
    g = synth._gen(7, dev)
    q = synth.randn_bf16((S, hq, D_QK), g, dev)
    k_new = synth.randn_bf16((S, hkv, D_QK), g, dev)
    v_new = synth.randn_bf16((S, hkv, D_V), g, dev)
    sink = synth.randn_f32((hq,), g, dev)
    cap = P + S + 256
    kc = torch.empty((1, hkv, cap, D_QK), dtype=torch.bfloat16, device=dev)
    vc = torch.empty((1, hkv, cap, D_V), dtype=torch.bfloat16, device=dev)
    for s0 in range(0, P, 4096):  # the prefix, written by the append kernel
        kp = synth.randn_bf16((1, 4096, hkv, D_QK), g, dev)
        vp = synth.randn_bf16((1, 4096, hkv, D_V), g, dev)
        ha.rope_kv_append(kp, vp, torch.tensor([s0], dtype=torch.int32, device=dev), kc, vc,
                          is_ring=False, rope_base=base)
    cu = torch.tensor([0, S], dtype=torch.int32, device=dev)
    pre = torch.tensor([P], dtype=torch.int32, device=dev)
    out = torch.empty((S, hq, D_V), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((S, hq), dtype=torch.float32, device=dev)
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    sptr = torch.cuda.current_stream(dev).cuda_stream

    def step():
        st = ha.hattn_prefill_cached(q, k_new, v_new, kc, vc, cu, pre, sink, out, lse, 1, S, S,
                                     P, cap, hq, hkv, D_QK, D_V, R, base, 0,
                                     1.0 / math.sqrt(D_QK), ws, ws.numel(), sptr)
        assert st == 0, ha.status_string(st)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ha.check_device_status()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        start.record()
        for _ in range(args.steps):
            step()
        stop.record()
        torch.cuda.synchronize()
    ha.check_device_status()
    ms = start.elapsed_time(stop) / args.steps
    hbm, tf_burst, tf_sust, src = measured_peaks()
    pairs = S * P + S * (S + 1) // 2
    flops = PAIR_FLOPS * hq * pairs
    byts = (S * (hq * D_QK * 2 + hkv * (D_QK + D_V) * 2 * 2 + hq * D_V * 2 + hq * 4)
            + P * hkv * (D_QK + D_V) * 2 + hq * 4)
    t = ms / 1e3
    tf, tf_name = tensor_peak(t, tf_burst, tf_sust)
    return {"metric": METRIC, "value": round(flops / t / 1e12, 3), "unit": "TFLOP/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 q/k/v, N(0,1) fp32 sinks)",
            "config": {"workload": "prefix_prefill: global layer (64q/4kv, base 5e6), 4096 new "
                                   "tokens over a cached prefix of 28672"},
            "roofline": {"bound": "tensor", "achieved": round(flops / t / 1e12, 2),
                         "peak": tf, "unit": "TFLOP/s",
                         "frac": round(flops / t / 1e12 / tf, 4), "traffic": None,
                         "peak_source": f"{src} {tf_name}"},
            "algorithmic": {"flops": flops, "bytes": byts}, "clocks": clk.summary()}


BWD_PAIR_FLOPS = 2 * (3 * D_QK + 2 * D_V)  # S, dQ, dK (192 deep) and dP, dV (128) per pair


def run_backward(args):
    """Backward of one window layer (64q/8kv, W 128, base 1e4) and one global
    layer (64q/4kv, base 5e6) over 32768 tokens each: hattn_prefill_backward
    per layer per step (the forward's out / lse are computed once, untimed)."""
    import global_attention_sinks_gqa_b300 as ha
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    sptr = torch.cuda.current_stream(dev).cuda_stream
    layers = []
    for name in ("swa_prefill_32k", "ga_prefill_32k"):
        p = synth.CONFIGS[name]
        c = synth.prefill_case(p["seqlens"], p["hq"], p["hkv"], window=p["window"],
                               rope_base=p["rope_base"], seed=p["seed"], device=dev)
        S = c.total
        g = synth.randn_bf16((S, c.hq, D_V), synth._gen(p["seed"] + 100, dev), dev)
        out, lse = ha.prefill(c.q, c.k, c.v, c.sink, c.cu_seqlens, max_seqlen=S,
                              window=c.window, rope_base=c.rope_base)
        ws = torch.empty(ha.hattn_prefill_backward_workspace_size(S, c.hq, c.hkv),
                         dtype=torch.uint8, device=dev)
        grads = (torch.empty_like(c.q), torch.empty_like(c.k), torch.empty_like(c.v),
                 torch.empty((c.hq,), dtype=torch.float32, device=dev))
        pairs = prefill_pairs(S, c.window)
        # read q, out, dout, lse, k, v; write dq, dk, dv
        byts = S * (c.hq * (2 * D_QK * 2 + 2 * D_V * 2 + 4) + c.hkv * 2 * (D_QK + D_V) * 2)
        layers.append(dict(name=name, c=c, g=g, out=out, lse=lse, ws=ws, grads=grads, S=S,
                           flops=BWD_PAIR_FLOPS * c.hq * pairs, bytes=byts))

    def run_layer(L):
        c, (dq, dk, dv, ds) = L["c"], L["grads"]
        st = ha.hattn_prefill_backward(c.q, c.k, c.v, c.sink, L["out"], L["lse"], L["g"], dq, dk,
                                       dv, ds, 1, c.cu_seqlens, L["S"], L["S"], c.hq, c.hkv, D_QK,
                                       D_V, R, c.rope_base, c.window, c.scale, L["ws"],
                                       L["ws"].numel(), sptr)
        assert st == 0, ha.status_string(st)

    for _ in range(args.warmup):
        for L in layers:
            run_layer(L)
    torch.cuda.synchronize()
    ha.check_device_status()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with ClockSampler(dev.index) as clk:
        for e in ev:
            e[0].record()
            run_layer(layers[0])
            e[1].record()
            run_layer(layers[1])
            e[2].record()
        torch.cuda.synchronize()
    ha.check_device_status()
    t_swa = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps / 1e3
    t_ga = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps / 1e3
    t = ev[0][0].elapsed_time(ev[-1][2]) / args.steps / 1e3
    hbm, tf_burst, tf_sust, src = measured_peaks()
    flops = sum(L["flops"] for L in layers)
    swa, ga = layers
    ga_tf = ga["flops"] / t_ga / 1e12
    tf_sust, tf_name = tensor_peak(t_ga, tf_burst, tf_sust)
    return {"metric": "prefill backward TFLOP/s (SWA+GA sink attention) vs B300 roofline",
            "value": round(flops / t / 1e12, 3), "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 q/k/v/dout, N(0,1) fp32 sinks)",
            "config": {"workload": "backward: one window layer (32768 tokens, 64q/8kv, W 128) "
                                   "and one global layer (32768 tokens, 64q/4kv)",
                       "flop_per_pair": BWD_PAIR_FLOPS},
            "roofline": {"bound": "tensor", "achieved": round(ga_tf, 2), "peak": tf_sust,
                         "unit": "TFLOP/s", "frac": round(ga_tf / tf_sust, 4), "traffic": None,
                         "kernel": "global layer backward (dK/dV + dQ kernels)",
                         "peak_source": f"{src} {tf_name}"},
            "parts": {"swa_backward": {"ms": round(t_swa * 1e3, 4),
                                       "GB/s": round(swa["bytes"] / t_swa / 1e9, 1),
                                       "frac_hbm": round(swa["bytes"] / t_swa / 1e9 / hbm, 4),
                                       "bytes": swa["bytes"]},
                      "ga_backward": {"ms": round(t_ga * 1e3, 4), "TFLOP/s": round(ga_tf, 2),
                                      "frac_tensor": round(ga_tf / tf_sust, 4),
                                      "peak": tf_name, "flops": ga["flops"]}},
            "gpu_launches": 8 * args.steps,  # prep, sink sum, dK/dV, dQ per layer
            "clocks": clk.summary()}


def run_paged_decode(args):
    """The global layer's decode step of the bench (batch 64 x 4 verify tokens,
    lengths U[8192, 65536]) over a paged copy of its cache: pages of 256
    positions in shuffled order, one hattn_decode_append_paged call per step."""
    import global_attention_sinks_gqa_b300 as ha
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl = Workload(dev)
    dd = [d for d in wl.dec if not d["ring"]][0]
    p = dd["p"]
    page = 256
    stride = (dd["cap"] + page - 1) // page
    kc, vc = dd["kc"], dd["vc"]
    B, hkv = wl.B, p["hkv"]
    num_pages = B * stride
    gen = torch.Generator(device="cpu")
    gen.manual_seed(11)
    table = torch.randperm(num_pages, generator=gen).to(torch.int32).reshape(B, stride).to(dev)
    kp = torch.empty((num_pages, hkv, page, D_QK), dtype=torch.bfloat16, device=dev)
    vp = torch.empty((num_pages, hkv, page, D_V), dtype=torch.bfloat16, device=dev)
    for b in range(B):
        for lp in range(stride):
            hi = min((lp + 1) * page, dd["cap"])
            kp[table[b, lp], :, :hi - lp * page] = kc[b, :, lp * page:hi]
            vp[table[b, lp], :, :hi - lp * page] = vc[b, :, lp * page:hi]
    del wl.layers
    ws_n = ha.hattn_decode_workspace_size(B, wl.T, p["hq"], hkv, D_V, wl.lmax, p["window"],
                                          stride * page, 0)
    ws = torch.empty(max(ws_n, 256), dtype=torch.uint8, device=dev)
    sptr = torch.cuda.current_stream(dev).cuda_stream

    def step():
        st = ha.hattn_decode_append_paged(dd["q"], dd["k_new"], dd["v_new"], kp, vp, table,
                                          stride, num_pages, page, dd["seqlens"], dd["sink"],
                                          dd["out"], dd["lse"], B, wl.T, p["hq"], hkv, D_QK,
                                          D_V, p["window"], wl.lmax, R, p["rope_base"],
                                          1.0 / math.sqrt(D_QK), ws, ws.numel(), sptr)
        assert st == 0, ha.status_string(st)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ha.check_device_status()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        start.record()
        for _ in range(args.steps):
            step()
        stop.record()
        torch.cuda.synchronize()
    ha.check_device_status()
    ms = start.elapsed_time(stop) / args.steps
    hbm, tf_burst, tf_sust, src = measured_peaks()
    byts = dd["bytes"] + dd["abytes"]
    gbs = byts / (ms / 1e3) / 1e9
    return {"metric": METRIC, "value": round(gbs, 1), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 q/k/v, N(0,1) fp32 sinks)",
            "config": {"workload": "paged_decode: global layer, batch 64 x 4 verify tokens, "
                                   "L ~ U[8192, 65536], pages of 256 positions, shuffled"},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm,
                         "unit": "GB/s", "frac": round(gbs / hbm, 4), "traffic": None,
                         "peak_source": f"{src} hbm_gbs"},
            "clocks": clk.summary()}


def run_profile_case(args):
    """One call of one part of the step at a chosen size, for an ncu capture:
    a warm-up call, then the profiled call inside the NVTX range "profile"."""
    import global_attention_sinks_gqa_b300 as ha
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    name = args.profile_case
    if name in ("swa_prefill", "ga_prefill"):
        c = synth.CONFIGS[name + "_32k"]
        S = args.seq or c["seqlens"][0]
        pc = synth.prefill_case([S], c["hq"], c["hkv"], window=c["window"],
                                rope_base=c["rope_base"], seed=c["seed"], device=dev)
        ws = torch.empty(ha.hattn_prefill_workspace_size(S, pc.hkv, D_QK), dtype=torch.uint8,
                         device=dev)

        def call():
            return ha.prefill(pc.q, pc.k, pc.v, pc.sink, pc.cu_seqlens, max_seqlen=S,
                              window=pc.window, rope_base=pc.rope_base,
                              softmax_scale=pc.scale, workspace=ws)
        work = f"{name} seq {S}"
    elif name in ("decode_swa", "decode_ga"):
        dc = synth.CONFIGS["decode_b64_t4"]
        kind = name.split("_")[1]
        p = dc[kind]
        B = args.batch or dc["B"]
        T = dc["T"]
        lens = synth.random_lengths(B, dc["lens"][0], dc["lens"][1], dc["seed"])
        cap = 131 if kind == "swa" else dc["lens"][1]
        kc = torch.randn((B, p["hkv"], cap, D_QK), device=dev).to(torch.bfloat16)
        vc = torch.randn((B, p["hkv"], cap, D_V), device=dev).to(torch.bfloat16)
        q = torch.randn((B, T, p["hq"], D_QK), device=dev).to(torch.bfloat16)
        sink = torch.randn(p["hq"], device=dev)
        sl = torch.tensor(lens, dtype=torch.int32, device=dev)

        def call():
            return ha.decode(q, kc, vc, sl, sink, max_seqlen_k=dc["lens"][1],
                             window=p["window"], is_ring=kind == "swa",
                             rope_base=p["rope_base"])
        work = f"{name} batch {B} x {T}"
    elif name in ("swa_backward", "ga_backward"):
        c = synth.CONFIGS[name.split("_")[0] + "_prefill_32k"]
        S = args.seq or c["seqlens"][0]
        pc = synth.prefill_case([S], c["hq"], c["hkv"], window=c["window"],
                                rope_base=c["rope_base"], seed=c["seed"], device=dev)
        g = synth.randn_bf16((S, pc.hq, D_V), synth._gen(c["seed"] + 100, dev), dev)
        out, lse = ha.prefill(pc.q, pc.k, pc.v, pc.sink, pc.cu_seqlens, max_seqlen=S,
                              window=pc.window, rope_base=pc.rope_base, softmax_scale=pc.scale)
        ws = torch.empty(ha.hattn_prefill_backward_workspace_size(S, pc.hq, pc.hkv),
                         dtype=torch.uint8, device=dev)

        def call():
            return ha.prefill_backward(pc.q, pc.k, pc.v, pc.sink, out, lse, g, pc.cu_seqlens,
                                       max_seqlen=S, window=pc.window, rope_base=pc.rope_base,
                                       softmax_scale=pc.scale, workspace=ws)
        work = f"{name} seq {S}"
    else:
        raise SystemExit(f"unknown profile case {name}")
    call()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("profile")
    call()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    ha.check_device_status()
    print(json.dumps({"profile_case": work, "ok": True}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--cpu-baseline", type=int, default=1)
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--extras", type=int, default=1,
                    help="also time the hybrid block at 256K and the backward after the step "
                         "(N = 1 only)")
    ap.add_argument("--launch-check", action="store_true",
                    help="with --gpus N: start the N ranks, meet at a barrier, take the max "
                         "over ranks and print one line (no attention work; checks the "
                         "replica launch)")
    ap.add_argument("--profile-case", default=None,
                    help="swa_prefill | ga_prefill | decode_swa | decode_ga | swa_backward | "
                         "ga_backward: one call, for ncu")
    ap.add_argument("--seq", type=int, default=0, help="prefill length for --profile-case")
    ap.add_argument("--batch", type=int, default=0, help="decode batch for --profile-case")
    ap.add_argument("--workload", default="step",
                    choices=["step", "hybrid_block_256k", "prefix_prefill", "paged_decode",
                             "backward"],
                    help="step: the default bench step; hybrid_block_256k: one hybrid block "
                         "(5 window + 1 global layer) over 262144 tokens; "
                         "prefix_prefill: 4096 new tokens over a cached 28672-token prefix; "
                         "paged_decode: the global decode step over a paged cache; "
                         "backward: the gradients of one window and one global layer")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args)
        return
    if args.workload == "hybrid_block_256k":
        print(json.dumps(run_hybrid_block(args)))
        return
    if args.workload == "backward":
        print(json.dumps(run_backward(args)))
        return
    if args.workload == "prefix_prefill":
        print(json.dumps(run_prefix_prefill(args)))
        return
    if args.workload == "paged_decode":
        print(json.dumps(run_paged_decode(args)))
        return
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # not started by a launcher: start one rank per GPU on this node
        sys.exit(launch_replicas(args.gpus, sys.argv[1:]))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    if args.launch_check:
        res = launch_check(rank, world)
    else:
        res = run_cuda(args, rank, world)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
