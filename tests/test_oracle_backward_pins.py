"""Pins of the backward oracle (CPU only).

The backward is the gradient of sum(dout * out) of the forward definition
(MiMo-V2-Flash paper review, section 3.2: the sink logit is a learnable
per-head parameter, so training needs its gradient next to those of q, k, v).
Nothing here compares the oracle with itself: the whole-matrix numpy backward
is pinned by central finite differences of the whole-matrix forward; the C
backward is checked against that, against torch autograd through its library
attention in the no-sink / no-RoPE special case, against finite differences of
the C forward in the sink, and against a closed form for the column sums of dv;
plus identities any correct backward keeps (a window covering the sequence is
global, packing restarts positions, a dominating sink zeroes every gradient).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
import synth


def _rand(shape, rng):
    return rng.standard_normal(shape)


def _brute_loss(q, k, v, sink, dout, cu, **kw):
    out, _ = brute.prefill(q, k, v, sink, cu, **kw)
    return float(np.sum(out * dout))


@pytest.mark.parametrize("window,rope_dim,seqlens", [(3, 4, [5, 3]), (0, 4, [6]), (2, 0, [4, 1])])
def test_brute_backward_matches_finite_differences(window, rope_dim, seqlens):
    rng = np.random.default_rng(11 + window)
    hq, hkv, dqk, dv = 4, 2, 8, 4
    total = sum(seqlens)
    cu = np.concatenate([[0], np.cumsum(seqlens)])
    q, k, v = _rand((total, hq, dqk), rng), _rand((total, hkv, dqk), rng), _rand((total, hkv, dv), rng)
    sink, dout = _rand((hq,), rng), _rand((total, hq, dv), rng)
    kw = dict(window=window, rope_base=100.0, scale=0.37, rope_dim=rope_dim)
    dq, dk, dvv, ds = brute.prefill_backward(q, k, v, sink, dout, cu, **kw)
    eps = 1e-5

    def fd(x, setter):
        g = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            x0 = x[idx]
            x[idx] = x0 + eps
            lp = setter()
            x[idx] = x0 - eps
            lm = setter()
            x[idx] = x0
            g[idx] = (lp - lm) / (2 * eps)
        return g

    loss = lambda: _brute_loss(q, k, v, sink, dout, cu, **kw)
    for x, got in ((q, dq), (k, dk), (v, dvv), (sink, ds)):
        ref = fd(x, loss)
        assert np.max(np.abs(ref - got)) < 1e-7, np.max(np.abs(ref - got))


@pytest.mark.parametrize("seqlens,hq,hkv,window,base,seed", [
    ([29], 8, 1, 16, 1e4, 21),
    ([40], 16, 1, 0, 5e6, 22),
    ([13, 27], 8, 4, 5, 1e4, 23),
    ([1, 2, 9], 4, 2, 2, 1e4, 24),
    ([33], 8, 8, 128, 1e4, 25),
])
def test_c_backward_matches_numpy_brute_force(seqlens, hq, hkv, window, base, seed):
    c = synth.prefill_case(seqlens, hq, hkv, window=window, rope_base=base, seed=seed)
    g = synth.randn_bf16((c.total, hq, 128), synth._gen(seed + 1, "cpu"), "cpu")
    kw = dict(window=window, rope_base=base, scale=c.scale)
    got = oracle.prefill_backward(c.q, c.k, c.v, c.sink, g, c.cu_seqlens.tolist(), **kw)
    ref = brute.prefill_backward(c.q, c.k, c.v, c.sink.double().numpy(), g,
                                 c.cu_seqlens.numpy(), **kw)
    for a, b in zip(got, ref):
        assert a.shape == b.shape
        assert np.max(np.abs(a - b)) < 1e-11 * max(1.0, np.max(np.abs(b)))


def test_backward_no_sink_no_rope_matches_torch_autograd():
    """Sink -> -inf and rope_dim = 0: textbook causal GQA attention, whose
    gradients torch autograd takes through scaled_dot_product_attention in fp64
    (the GQA replication of K/V heads inside the graph sums dk, dv over the
    query heads of a group)."""
    S, hq, hkv = 48, 8, 2
    c = synth.prefill_case([S], hq, hkv, window=0, rope_base=1e4, seed=31)
    g = synth.randn_bf16((S, hq, 128), synth._gen(32, "cpu"), "cpu")
    sink = torch.full((hq,), -math.inf)
    for window in (0, 7):
        dq, dk, dvv, ds = oracle.prefill_backward(c.q, c.k, c.v, sink, g, [0, S], window=window,
                                                  rope_base=1e4, scale=c.scale, rope_dim=0)
        q = c.q.double().requires_grad_()
        k = c.k.double().requires_grad_()
        v = c.v.double().requires_grad_()
        qt = q.transpose(0, 1)[None]
        kt = k.repeat_interleave(hq // hkv, dim=1).transpose(0, 1)[None]
        vt = v.repeat_interleave(hq // hkv, dim=1).transpose(0, 1)[None]
        i = torch.arange(S)[:, None]
        j = torch.arange(S)[None, :]
        mask = (j <= i) & ((i - j < window) if window else True)
        out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                               scale=c.scale)
        (out[0].transpose(0, 1) * g.double()).sum().backward()
        assert np.max(np.abs(dq - q.grad.numpy())) < 1e-11
        assert np.max(np.abs(dk - k.grad.numpy())) < 1e-11
        assert np.max(np.abs(dvv - v.grad.numpy())) < 1e-11
        assert np.all(ds == 0.0)


def test_sink_gradient_matches_finite_differences_of_the_c_forward():
    """The C forward takes the sink in double, so its derivative in each sink
    logit is available by central differences at full head dims."""
    seqlens, hq, hkv, window = [37, 20], 8, 2, 16
    c = synth.prefill_case(seqlens, hq, hkv, window=window, rope_base=1e4, seed=41)
    g = synth.randn_bf16((c.total, hq, 128), synth._gen(42, "cpu"), "cpu")
    cu = c.cu_seqlens.tolist()
    kw = dict(window=window, rope_base=1e4, scale=c.scale)
    _, _, _, ds = oracle.prefill_backward(c.q, c.k, c.v, c.sink, g, cu, **kw)
    gd = g.double().numpy()
    eps = 1e-5
    for h in range(hq):
        s = c.sink.double().numpy().copy()
        s[h] += eps
        op, _ = oracle.prefill(c.q, c.k, c.v, s, cu, **kw)
        s[h] -= 2 * eps
        om, _ = oracle.prefill(c.q, c.k, c.v, s, cu, **kw)
        ref = (np.sum(op * gd) - np.sum(om * gd)) / (2 * eps)
        assert abs(ref - ds[h]) < 1e-7 * max(1.0, abs(ref)), (h, ref, ds[h])


def test_dv_column_sums_closed_form():
    """Each row's key weights sum to 1 - p_sink, so the sum of dv over a KV
    head's keys is sum over its rows and query heads of (1 - e^(sink - lse)) dout."""
    seqlens, hq, hkv, window = [50, 11], 8, 2, 9
    c = synth.prefill_case(seqlens, hq, hkv, window=window, rope_base=1e4, seed=51)
    g = synth.randn_bf16((c.total, hq, 128), synth._gen(52, "cpu"), "cpu")
    cu = c.cu_seqlens.tolist()
    kw = dict(window=window, rope_base=1e4, scale=c.scale)
    _, _, dvv, _ = oracle.prefill_backward(c.q, c.k, c.v, c.sink, g, cu, **kw)
    _, lse = oracle.prefill(c.q, c.k, c.v, c.sink, cu, **kw)
    w = 1.0 - np.exp(c.sink.double().numpy()[None, :] - lse)           # [total, hq]
    gd = g.double().numpy()
    G = hq // hkv
    for b in range(len(seqlens)):
        a, e = cu[b], cu[b + 1]
        for kv in range(hkv):
            ref = np.einsum("th,thd->d", w[a:e, kv * G:(kv + 1) * G], gd[a:e, kv * G:(kv + 1) * G])
            assert np.max(np.abs(dvv[a:e, kv].sum(0) - ref)) < 1e-10


def test_planted_backward_mistakes_are_caught():
    """Backwards with a plausible mistake (the sink dropped from the
    denominator, dk' not turned back) fail the finite-difference pin."""
    rng = np.random.default_rng(7)
    hq, hkv, dqk, dv, S = 2, 1, 8, 4, 5
    q, k, v = _rand((S, hq, dqk), rng), _rand((S, hkv, dqk), rng), _rand((S, hkv, dv), rng)
    sink, dout = _rand((hq,), rng), _rand((S, hq, dv), rng)
    cu = np.array([0, S])
    kw = dict(window=0, rope_base=100.0, scale=0.37, rope_dim=4)
    eps = 1e-5
    ref_dk = np.zeros_like(k)
    for idx in np.ndindex(k.shape):
        k0 = k[idx]
        k[idx] = k0 + eps
        lp = _brute_loss(q, k, v, sink, dout, cu, **kw)
        k[idx] = k0 - eps
        lm = _brute_loss(q, k, v, sink, dout, cu, **kw)
        k[idx] = k0
        ref_dk[idx] = (lp - lm) / (2 * eps)
    no_sink = brute.prefill_backward(q, k, v, np.full(hq, -np.inf), dout, cu, **kw)[1]
    assert np.max(np.abs(no_sink - ref_dk)) > 1e-3
    # dk' left rotated: apply the forward rotation once more instead of undoing it
    dk = brute.prefill_backward(q, k, v, sink, dout, cu, **kw)[1]
    pos = np.arange(S)
    twice = np.transpose(brute.rope_complex(brute.rope_complex(np.transpose(dk, (1, 0, 2)), pos,
                                                               100.0, 4), pos, 100.0, 4), (1, 0, 2))
    assert np.max(np.abs(twice - ref_dk)) > 1e-3
    assert np.max(np.abs(dk - ref_dk)) < 1e-7


def test_backward_window_covering_the_sequence_equals_global():
    c = synth.prefill_case([45], 8, 2, window=45, rope_base=1e4, seed=71)
    g = synth.randn_bf16((45, 8, 128), synth._gen(72, "cpu"), "cpu")
    a = oracle.prefill_backward(c.q, c.k, c.v, c.sink, g, [0, 45], window=45, rope_base=1e4,
                                scale=c.scale)
    b = oracle.prefill_backward(c.q, c.k, c.v, c.sink, g, [0, 45], window=0, rope_base=1e4,
                                scale=c.scale)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_backward_packing_restarts_positions():
    """A packed batch equals its sequences run one by one (positions restart at
    0 in each); the sink gradient is their sum."""
    lens = [17, 30]
    c = synth.prefill_case(lens, 8, 4, window=9, rope_base=1e4, seed=73)
    g = synth.randn_bf16((47, 8, 128), synth._gen(74, "cpu"), "cpu")
    kw = dict(window=9, rope_base=1e4, scale=c.scale)
    packed = oracle.prefill_backward(c.q, c.k, c.v, c.sink, g, [0, 17, 47], **kw)
    parts = [oracle.prefill_backward(c.q[a:e], c.k[a:e], c.v[a:e], c.sink, g[a:e], [0, e - a],
                                     **kw) for a, e in ((0, 17), (17, 47))]
    for i in range(3):
        ref = np.concatenate([p[i] for p in parts], 0)
        assert np.max(np.abs(packed[i] - ref)) < 1e-12
    assert np.max(np.abs(packed[3] - (parts[0][3] + parts[1][3]))) < 1e-12


def test_backward_vanishes_as_the_sink_dominates():
    """With a sink logit far above every key's, the keys' weights and the output
    go to 0, and with them every gradient (the sink's: -p_sink (dout . out))."""
    c = synth.prefill_case([25], 4, 2, window=0, rope_base=1e4, seed=75)
    g = synth.randn_bf16((25, 4, 128), synth._gen(76, "cpu"), "cpu")
    for s in (40.0, 80.0):
        sink = torch.full((4,), s)
        dq, dk, dv, ds = oracle.prefill_backward(c.q, c.k, c.v, sink, g, [0, 25], window=0,
                                                 rope_base=1e4, scale=c.scale)
        bound = 1e3 * math.exp(-(s - 10.0))
        for x in (dq, dk, dv, ds):
            assert np.max(np.abs(x)) < bound, (s, np.max(np.abs(x)))
