"""Pins for the fp64 CPU oracle: facts the pages and the mathematics fix.

Each test checks the oracle against something other than itself -- a second
brute-force formulation, a library routine, a closed form or an identity --
chosen so that a dropped term, a wrong sign or index, or a transposed operand
fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def _case(seqlens, hq, hkv, window, base, seed, dqk=192, dv=128, sink_mean=0.0, sink_std=1.0):
    return synth.prefill_case(seqlens, hq, hkv, window=window, rope_base=base, seed=seed,
                              dqk=dqk, dv=dv, sink_mean=sink_mean, sink_std=sink_std)


def _oracle_prefill(c, **kw):
    kw.setdefault("window", c.window)
    kw.setdefault("rope_base", c.rope_base)
    kw.setdefault("scale", c.scale)
    return oracle.prefill(c.q, c.k, c.v, c.sink, c.cu_seqlens.tolist(), **kw)


@pytest.mark.parametrize("seqlens,hq,hkv,window,base,seed", [
    ([37], 8, 1, 16, 1e4, 1),
    ([64], 16, 1, 0, 5e6, 2),
    ([23, 41], 8, 8, 7, 1e4, 3),
    ([50], 4, 2, 128, 1e4, 4),
    ([1, 2, 3], 2, 1, 2, 1e4, 5),
])
def test_c_oracle_matches_numpy_brute_force(seqlens, hq, hkv, window, base, seed):
    c = _case(seqlens, hq, hkv, window, base, seed)
    o1, l1 = _oracle_prefill(c)
    o2, l2 = brute.prefill(c.q, c.k, c.v, c.sink.double().numpy(), c.cu_seqlens.numpy(),
                           window=window, rope_base=base, scale=c.scale)
    assert np.max(np.abs(o1 - o2)) < 1e-12
    assert np.max(np.abs(l1 - l2)) < 1e-12


def test_worked_example_golden():
    """Hand-derived two-token example (tests/golden/worked_example.json)."""
    with open(os.path.join(HERE, "golden", "worked_example.json")) as f:
        g = json.load(f)
    inp = g["inputs"]
    q = torch.tensor(inp["q"], dtype=torch.bfloat16)
    k = torch.tensor(inp["k"], dtype=torch.bfloat16)
    v = torch.tensor(inp["v"], dtype=torch.bfloat16)
    env = {"e": math.e, "exp": math.exp, "cos": math.cos, "log": math.log}
    for s in inp["sinks"]:
        for case in g["cases"]:
            out, lse = oracle.prefill(q, k, v, [s], [0, 2], window=case["window"],
                                      rope_base=inp["rope_base"], scale=inp["scale"],
                                      rope_dim=inp["rope_dim"])
            env["s"] = s
            want_o = np.array([[eval(x, {}, env) for x in row] for row in case["out"]])
            want_l = np.array([eval(x, {}, env) for x in case["lse"]])
            assert np.max(np.abs(out[:, 0, :] - want_o)) < 1e-14
            assert np.max(np.abs(lse[:, 0] - want_l)) < 1e-14


def test_window_not_below_seqlen_equals_global():
    c = _case([90], 8, 2, 0, 1e4, 11)
    og, lg = _oracle_prefill(c, window=0)
    for w in (90, 91, 1000):
        ow, lw = _oracle_prefill(c, window=w)
        assert np.array_equal(og, ow) and np.array_equal(lg, lw)
    o89, _ = _oracle_prefill(c, window=89)
    assert np.max(np.abs(o89[-1] - og[-1])) > 1e-6  # the last row loses key 0


def test_no_sink_no_rope_matches_torch_sdpa():
    """s_sink -> -inf and rope_dim = 0 reduce to textbook causal GQA softmax
    attention, checked against torch's scaled_dot_product_attention in fp64."""
    c = _case([70], 8, 2, 0, 1e4, 12)
    sink = torch.full((8,), -math.inf)
    for window in (0, 9):
        out, lse = oracle.prefill(c.q, c.k, c.v, sink, [0, 70], window=window, rope_base=1e4,
                                  scale=c.scale, rope_dim=0)
        q = c.q.double().transpose(0, 1)[None]                  # [1, hq, S, d]
        k = c.k.double().repeat_interleave(4, dim=1).transpose(0, 1)[None]
        v = c.v.double().repeat_interleave(4, dim=1).transpose(0, 1)[None]
        i = torch.arange(70)[:, None]
        j = torch.arange(70)[None, :]
        mask = (j <= i) & ((i - j < window) if window else True)
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask,
                                                               scale=c.scale)
        ref = ref[0].transpose(0, 1).numpy()
        assert np.max(np.abs(out - ref)) < 1e-12
        logits = (q @ k.transpose(-1, -2)) * c.scale
        logits = logits.masked_fill(~mask, -math.inf)
        ref_lse = torch.logsumexp(logits, dim=-1)[0].transpose(0, 1).numpy()
        assert np.max(np.abs(lse - ref_lse)) < 1e-12


def test_sink_closed_form():
    """out_s = out_nosink * sigmoid(lse_nosink - s), lse_s = logaddexp(lse_nosink, s)."""
    c = _case([40, 25], 8, 1, 12, 1e4, 13)
    o0, l0 = oracle.prefill(c.q, c.k, c.v, torch.full((8,), -math.inf), c.cu_seqlens.tolist(),
                            window=12, rope_base=1e4, scale=c.scale)
    s = c.sink.double().numpy()
    o1, l1 = _oracle_prefill(c)
    sig = 1.0 / (1.0 + np.exp(-(l0 - s[None, :])))
    assert np.max(np.abs(o1 - o0 * sig[:, :, None])) < 1e-13
    assert np.max(np.abs(l1 - np.logaddexp(l0, s[None, :]))) < 1e-12


def test_large_sink_drives_output_to_zero():
    c = _case([33], 4, 1, 0, 1e4, 14)
    out, lse = oracle.prefill(c.q, c.k, c.v, torch.full((4,), 60.0), [0, 33], window=0,
                              rope_base=1e4, scale=c.scale)
    assert np.max(np.abs(out)) < 1e-16
    assert np.max(np.abs(lse - 60.0)) < 1e-12


def test_gqa_equals_replicated_kv_heads():
    c = _case([48], 16, 2, 20, 1e4, 15)
    o1, l1 = _oracle_prefill(c)
    k_rep = c.k.repeat_interleave(8, dim=1)
    v_rep = c.v.repeat_interleave(8, dim=1)
    o2, l2 = oracle.prefill(c.q, k_rep, v_rep, c.sink, [0, 48], window=20, rope_base=1e4,
                            scale=c.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # and a swapped head-to-group map would differ
    k_swap = torch.flip(c.k, dims=[1])
    v_swap = torch.flip(c.v, dims=[1])
    o3, _ = oracle.prefill(c.q, k_swap, v_swap, c.sink, [0, 48], window=20, rope_base=1e4,
                           scale=c.scale)
    assert np.max(np.abs(o3 - o1)) > 1e-3


def test_zero_query_closed_form():
    """q = 0 makes every logit 0: out_p = sum of the n_p visible values / (n_p + e^s),
    n_p = min(p + 1, W); this pins the window's width (W keys including the
    query), causality and the sink's place in the denominator."""
    S, W = 300, 128
    c = _case([S], 2, 1, W, 1e4, 16)
    q0 = torch.zeros_like(c.q)
    out, lse = oracle.prefill(q0, c.k, c.v, c.sink, [0, S], window=W, rope_base=1e4,
                              scale=c.scale)
    v = c.v.double().numpy()[:, 0, :]
    cs = np.concatenate([np.zeros((1, v.shape[1])), np.cumsum(v, axis=0)], 0)
    p = np.arange(S)
    lo = np.maximum(0, p - W + 1)
    n = p - lo + 1
    sums = cs[p + 1] - cs[lo]
    for h in range(2):
        s = float(c.sink[h])
        want = sums / (n + math.exp(s))[:, None]
        assert np.max(np.abs(out[:, h, :] - want)) < 1e-12
        assert np.max(np.abs(lse[:, h] - np.log(n + math.exp(s)))) < 1e-12


def test_rope_closed_forms():
    """Half-split RoPE: e_i at position p turns into (cos p*th_i, sin p*th_i) on
    dims (i, i+32); position 0 is the identity; dims 64.. pass through; norms
    are kept; the logit depends only on the position difference."""
    base, R, D = 1e4, 64, 192
    eye = torch.zeros((32, D), dtype=torch.bfloat16)
    for i in range(32):
        eye[i, i] = 1.0
    for p in (0, 1, 7, 262143):
        y = oracle.rope(eye, [p] * 32, rope_base=base, rope_dim=R)
        for i in range(32):
            th = base ** (-2.0 * i / R)
            assert abs(y[i, i] - math.cos(p * th)) < 1e-12
            assert abs(y[i, i + 32] - math.sin(p * th)) < 1e-12
            y[i, i] = 0.0
            y[i, i + 32] = 0.0
        assert np.max(np.abs(y)) == 0.0
    g = torch.Generator().manual_seed(17)
    x = torch.randn((6, D), generator=g).to(torch.bfloat16)
    xd = x.double().numpy()
    y0 = oracle.rope(x, [0] * 6, rope_base=base)
    assert np.array_equal(y0, xd)
    y = oracle.rope(x, [5, 77, 1000, 65535, 131071, 262143], rope_base=5e6)
    assert np.array_equal(y[:, 64:], xd[:, 64:])
    assert np.max(np.abs(np.linalg.norm(y, axis=1) - np.linalg.norm(xd, axis=1))) < 1e-12
    # relative position: <R(p) q, R(j) k> == <R(p + d) q, R(j + d) k>
    qv, kv = x[:3], x[3:]
    for d in (1, 1000, 200000):
        a = oracle.rope(qv, [10, 500, 3], rope_base=base)
        b = oracle.rope(kv, [4, 499, 3], rope_base=base)
        a2 = oracle.rope(qv, [10 + d, 500 + d, 3 + d], rope_base=base)
        b2 = oracle.rope(kv, [4 + d, 499 + d, 3 + d], rope_base=base)
        assert np.max(np.abs((a * b).sum(1) - (a2 * b2).sum(1))) < 1e-9
    # the complex-rotation form of brute.py agrees
    yb = brute.rope_complex(xd, np.array([5, 77, 1000, 65535, 131071, 262143]), 5e6, 64)
    assert np.max(np.abs(yb - y)) < 1e-12


def test_varlen_packing_restarts_positions():
    c = _case([30, 45, 17], 8, 2, 10, 1e4, 18)
    o, l = _oracle_prefill(c)
    a = 0
    for L in c.seqlens:
        os_, ls_ = oracle.prefill(c.q[a:a + L], c.k[a:a + L], c.v[a:a + L], c.sink, [0, L],
                                  window=10, rope_base=1e4, scale=c.scale)
        assert np.array_equal(o[a:a + L], os_) and np.array_equal(l[a:a + L], ls_)
        a += L


def test_row_sampling_equals_full():
    c = _case([60, 40], 8, 1, 0, 5e6, 19)
    o, l = _oracle_prefill(c)
    rows = [0, 17, 59, 60, 99, 61]
    os_, ls_ = _oracle_prefill(c, rows=rows)
    assert np.array_equal(o[rows], os_) and np.array_equal(l[rows], ls_)


@pytest.mark.parametrize("window,T", [(0, 4), (16, 4), (16, 1), (5, 3)])
def test_decode_equals_prefill_last_rows(window, T):
    lens = [40, 21, 33]
    d = synth.decode_case(lens, T, 8, 2, window=window, rope_base=1e4, seed=20)
    out, lse = oracle.decode(d.q, d.k_hist, d.v_hist, lens, d.sink, window=window,
                             rope_base=1e4, scale=d.scale)
    g = torch.Generator().manual_seed(21)
    for b, L in enumerate(lens):
        qf = torch.randn((L, 8, 192), generator=g).to(torch.bfloat16)
        qf[L - T:] = d.q[b]
        po, pl = oracle.prefill(qf, d.k_hist[b, :L], d.v_hist[b, :L], d.sink, [0, L],
                                window=window, rope_base=1e4, scale=d.scale,
                                rows=list(range(L - T, L)))
        assert np.max(np.abs(po - out[b])) < 1e-13
        assert np.max(np.abs(pl - lse[b])) < 1e-13


def test_split_merge_identity():
    """Partial (out_i, lse_i) over disjoint key ranges without the sink, merged by
    log-sum-exp with the sink added once, equal the unsplit result."""
    lens = [90, 64]
    for window in (0, 20):
        d = synth.decode_case(lens, 4, 8, 1, window=window, rope_base=5e6, seed=22)
        kw = dict(window=window, rope_base=5e6, scale=d.scale)
        full_o, full_l = oracle.decode(d.q, d.k_hist, d.v_hist, lens, d.sink, **kw)
        edges = [0, 13, 50, 71, -1]
        parts = [oracle.decode(d.q, d.k_hist, d.v_hist, lens, d.sink, key_lo=a, key_hi=b,
                               sink_on=False, **kw) for a, b in zip(edges[:-1], edges[1:])]
        s = d.sink.double().numpy()[None, None, :]
        lses = np.stack([p[1] for p in parts] + [np.broadcast_to(s, full_l.shape)], 0)
        lse = np.logaddexp.reduce(lses, axis=0)
        out = sum(np.exp(p[1] - lse)[..., None] * p[0] for p in parts)
        assert np.max(np.abs(out - full_o)) < 1e-13
        assert np.max(np.abs(lse - full_l)) < 1e-12


def test_decode_matches_brute_force_at_positions():
    lens = [29, 50]
    T = 3
    d = synth.decode_case(lens, T, 4, 1, window=8, rope_base=1e4, seed=23)
    out, lse = oracle.decode(d.q, d.k_hist, d.v_hist, lens, d.sink, window=8, rope_base=1e4,
                             scale=d.scale)
    for b, L in enumerate(lens):
        o2, l2 = brute.attention_one_sequence(
            brute.bf16_to_f64(d.q[b]), brute.bf16_to_f64(d.k_hist[b, :L]),
            brute.bf16_to_f64(d.v_hist[b, :L]), d.sink.double().numpy(), window=8,
            rope_base=1e4, scale=d.scale, q_pos=np.arange(L - T, L))
        assert np.max(np.abs(o2 - out[b])) < 1e-12
        assert np.max(np.abs(l2 - lse[b])) < 1e-12


def test_planted_mistakes_are_caught():
    """A mistake planted in a copy of the brute force (wrong RoPE sign, window
    off by one, sink dropped) must disagree with the C oracle."""
    c = _case([60], 8, 1, 16, 1e4, 24)
    o, _ = _oracle_prefill(c)
    qd, kd, vd = (brute.bf16_to_f64(t) for t in (c.q, c.k, c.v))
    s = c.sink.double().numpy()

    def run(**kw):
        return brute.attention_one_sequence(qd, kd, vd, s, rope_base=1e4, scale=c.scale, **kw)[0]

    assert np.max(np.abs(run(window=16) - o)) < 1e-12
    assert np.max(np.abs(run(window=17) - o)) > 1e-4            # window off by one
    assert np.max(np.abs(run(window=15) - o)) > 1e-4
    ob = brute.attention_one_sequence(qd, kd, vd, np.full(8, -np.inf), window=16,
                                      rope_base=1e4, scale=c.scale)[0]
    assert np.max(np.abs(ob - o)) > 1e-4                        # sink dropped
    flip = qd.copy()
    flip[:, :, 32:64] *= -1
    kflip = kd.copy()
    kflip[:, :, 32:64] *= -1                                    # rotation sign reversed
    of = brute.attention_one_sequence(flip, kflip, vd, s, window=16, rope_base=1e4,
                                      scale=c.scale)[0]
    assert np.max(np.abs(of - o)) > 1e-4
