"""Parity of hattn_prefill_backward against the fp64 oracle (B300 only).

Inputs are seeded N(0, 1) bf16 tensors (the recipe of the forward tests);
out and lse come from the CUDA forward, as they would in training.  The
oracle recomputes everything in fp64 from q, k, v, sink and dout.

Tolerance (derived from the arithmetic, not fitted): each gradient is a sum
of products whose factors are rounded to bf16 once (P, dS, the rotated dims;
relative error 2^-9 each), accumulated in fp32, and the result is rounded to
bf16 (2^-9).  Independent rounding errors of relative size ~2^-8 per term
give a relative L2 error of a few 1e-3; the bound is 1e-2 on the relative L2
error and 4e-2 of the largest reference magnitude element-wise.  The sink
gradient is an fp32 sum of per-row terms -e^(sink - lse) (dout . out) whose
out is the forward's bf16 output (its error, a few 1e-3 relative, enters
every term): bound 1e-2 of the sum of the terms' absolute values.
"""
import math

import numpy as np
import pytest
import torch

import global_attention_sinks_gqa_b300 as ha
import oracle
import synth

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
MAX_ABS = 4e-2


def _rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _run(seqlens, hq, hkv, window, base, seed, dout_seed=None, sink_mean=0.0, sink_std=1.0):
    dev = torch.device("cuda")
    c = synth.prefill_case(seqlens, hq, hkv, window=window, rope_base=base, seed=seed,
                           sink_mean=sink_mean, sink_std=sink_std)
    total = c.total
    g = synth.randn_bf16((total, hq, 128), synth._gen(seed + 1000 if dout_seed is None
                                                      else dout_seed, "cpu"), "cpu")
    q, k, v, sink = c.q.to(dev), c.k.to(dev), c.v.to(dev), c.sink.to(dev)
    cu = c.cu_seqlens.to(dev)
    S = max(seqlens)
    out, lse = ha.prefill(q, k, v, sink, cu, max_seqlen=S, window=window, rope_base=base)
    dq, dk, dv, ds = ha.prefill_backward(q, k, v, sink, out, lse, g.to(dev), cu, max_seqlen=S,
                                         window=window, rope_base=base)
    torch.cuda.synchronize()
    ha.check_device_status()
    ref = oracle.prefill_backward(c.q, c.k, c.v, c.sink, g, c.cu_seqlens.tolist(), window=window,
                                  rope_base=base, scale=c.scale)
    return (dq.double().cpu().numpy(), dk.double().cpu().numpy(), dv.double().cpu().numpy(),
            ds.double().cpu().numpy()), ref, (c, g, out, lse)


def _check(got, ref, what, extra):
    errs = {}
    for name, a, b in zip(("dq", "dk", "dv"), got[:3], ref[:3]):
        assert np.all(np.isfinite(a)), (what, name)
        r = _rel_l2(a, b)
        m = float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))
        errs[name] = (r, m)
        assert r < REL_L2 and m < MAX_ABS, (what, name, r, m)
    # the sink gradient's error comes from delta = dout . out taken with the
    # forward's bf16 out; it is bounded against the sum of the terms' sizes
    c, g, out, lse = extra
    ps = torch.exp(c.sink.double()[None, :] - lse.double().cpu())
    mag = (ps * (g.double() * out.double().cpu()).sum(-1)).abs().sum(0).numpy()
    ds, dsr = got[3], ref[3]
    assert np.all(np.abs(ds - dsr) <= 1e-2 * mag + 1e-4), (what, ds, dsr, mag)
    return errs


@pytest.mark.parametrize("seqlens,hq,hkv,window,base,seed", [
    ([300, 77], 16, 2, 128, 1e4, 1),          # window, G = 8, ragged tails
    ([513], 64, 8, 128, 1e4, 2),              # the window layer's heads, several key blocks
    ([260], 32, 2, 0, 5e6, 3),                # global, G = 16
    ([200, 1, 64], 64, 4, 0, 5e6, 4),         # the global layer's heads, a one-token sequence
    ([150], 4, 4, 0, 1e4, 5),                 # G = 1
    ([190, 33], 8, 4, 16, 1e4, 6),            # G = 2, short window
    ([129], 16, 4, 5, 1e4, 7),                # G = 4, window 5
    ([0, 90, 0], 16, 2, 128, 1e4, 8),         # empty sequences around one
])
def test_backward_matches_oracle(seqlens, hq, hkv, window, base, seed):
    got, ref, extra = _run(seqlens, hq, hkv, window, base, seed)
    errs = _check(got, ref, (seqlens, hq, hkv, window), extra)
    print(seqlens, hq, hkv, window, {k: (f"{r:.2e}", f"{m:.2e}") for k, (r, m) in errs.items()})


@pytest.mark.parametrize("seqlens,hq,hkv,window,sink_mean,sink_std,seed", [
    ([140, 9], 16, 2, 1, 0.0, 1.0, 11),      # W = 1: each query sees only itself
    ([300], 16, 2, 128, 8.0, 2.0, 12),       # heavy sinks: the sink takes most of the weight
    ([260], 32, 2, 0, 6.0, 2.0, 13),
])
def test_backward_degenerate_and_heavy_sinks(seqlens, hq, hkv, window, sink_mean, sink_std,
                                             seed):
    base = 1e4 if window else 5e6
    got, ref, extra = _run(seqlens, hq, hkv, window, base, seed, sink_mean=sink_mean,
                           sink_std=sink_std)
    _check(got, ref, (seqlens, hq, hkv, window, sink_mean), extra)


def test_backward_is_deterministic():
    dev = torch.device("cuda")
    c = synth.prefill_case([700], 16, 2, window=0, rope_base=5e6, seed=9, device=dev)
    g = synth.randn_bf16((700, 16, 128), synth._gen(10, dev), dev)
    out, lse = ha.prefill(c.q, c.k, c.v, c.sink, c.cu_seqlens, max_seqlen=700, window=0,
                          rope_base=5e6)
    a = ha.prefill_backward(c.q, c.k, c.v, c.sink, out, lse, g, c.cu_seqlens, max_seqlen=700,
                            window=0, rope_base=5e6)
    b = ha.prefill_backward(c.q, c.k, c.v, c.sink, out, lse, g, c.cu_seqlens, max_seqlen=700,
                            window=0, rope_base=5e6)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("window,hkv,base", [(128, 8, 1e4), (0, 4, 5e6)])
def test_backward_full_size_closed_forms(window, hkv, base):
    """One 32768-token layer with the model's heads: dv's sum over each KV
    head's keys equals sum over its rows of (1 - e^(sink - lse)) dout (each
    row's key weights sum to 1 - p_sink), and the sink gradient equals
    -sum e^(sink - lse) (dout . out); both evaluated in fp64 from the
    forward's out / lse."""
    dev = torch.device("cuda")
    S, hq = 32768, 64
    G = hq // hkv
    c = synth.prefill_case([S], hq, hkv, window=window, rope_base=base, seed=77, device=dev)
    g = synth.randn_bf16((S, hq, 128), synth._gen(78, dev), dev)
    out, lse = ha.prefill(c.q, c.k, c.v, c.sink, c.cu_seqlens, max_seqlen=S, window=window,
                          rope_base=base)
    dq, dk, dv, ds = ha.prefill_backward(c.q, c.k, c.v, c.sink, out, lse, g, c.cu_seqlens,
                                         max_seqlen=S, window=window, rope_base=base)
    torch.cuda.synchronize()
    ha.check_device_status()
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    ps = torch.exp(c.sink.double()[None, :] - lse.double())             # [S, hq]
    w = (1.0 - ps)[:, :, None] * g.double()
    ref = w.view(S, hkv, G, 128).sum(dim=(0, 2))                          # [hkv, 128]
    got = dv.double().sum(dim=0)
    scale = w.abs().view(S, hkv, G, 128).sum(dim=(0, 2))
    assert torch.all((got - ref).abs() <= 2e-2 * scale.clamp_min(1.0)), \
        float(((got - ref).abs() / scale.clamp_min(1.0)).max())
    delta = (g.double() * out.double()).sum(-1)
    ref_ds = -(ps * delta).sum(0)
    mag = (ps * delta).abs().sum(0)
    assert torch.all((ds.double() - ref_ds).abs() <= 1e-3 * mag + 1e-3)
