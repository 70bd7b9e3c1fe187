"""Device-side checks of the sequence offsets (cu_seqlens, prefix lengths).

The offsets live in device memory, where the host cannot read them before
the launch; the kernels check each sequence's slice of the packed rows and
skip a sequence whose slice is not inside [0, total_tokens), is longer than
max_seqlen, or (cached prefill) runs past the cache, recording
HATTN_ERR_INVALID_ARG.  Each test hands the kernels such offsets with output
buffers that have slack rows past total_tokens filled with a sentinel: the
sentinel must survive (nothing is written past the outputs), the status must
be reported, and the sequences with valid offsets must still match the
oracle.  Every access stays inside allocated memory, so nothing can fault.
"""
import numpy as np
import pytest
import torch

import global_attention_sinks_gqa_b300 as ha
import oracle
import synth
from gpu_util import compare

pytestmark = pytest.mark.gpu

SLACK = 256
SENTINEL = 7.0


def _slack(shape, dtype, dev):
    return torch.full((shape[0] + SLACK, *shape[1:]), SENTINEL, dtype=dtype, device=dev)


# (offsets, max_seqlen, (a valid sequence, how many of its first rows no
# other valid sequence also writes)); total_tokens is 300 in every case
CASES = [
    ([0, 100, 400], 300, (0, 100)),        # the last sequence runs past total_tokens
    ([0, 50, 300], 200, (0, 50)),          # a sequence longer than max_seqlen
    ([0, 200, 100, 300], 200, (0, 100)),   # decreasing offsets (a negative length); the
                                           # third sequence overlaps rows 100..199
    ([-50, 100, 300], 200, (1, 200)),      # a negative first offset
]


@pytest.mark.parametrize("window,base", [(128, 1e4), (0, 5e6)])
@pytest.mark.parametrize("cu,max_seqlen,good", CASES)
def test_prefill_skips_and_reports_bad_offsets(cu, max_seqlen, good, window, base):
    dev = torch.device("cuda")
    total, G = 300, 8
    c = synth.prefill_case([total], 2 * G, 2, window=window, rope_base=base, seed=901)
    q, k, v, sink = c.q.to(dev), c.k.to(dev), c.v.to(dev), c.sink.to(dev)
    out_full = _slack((total, c.hq, 128), torch.bfloat16, dev)
    lse_full = _slack((total, c.hq), torch.float32, dev)
    cu_d = torch.tensor(cu, dtype=torch.int32, device=dev)
    ha.prefill(q, k, v, sink, cu_d, max_seqlen=max_seqlen, window=window, rope_base=base,
               out=out_full[:total], lse=lse_full[:total])
    torch.cuda.synchronize()
    assert ha.hattn_check_device_status() == ha.HATTN_ERR_INVALID_ARG
    assert bool((out_full[total:] == SENTINEL).all()), "rows past total_tokens were written"
    assert bool((lse_full[total:] == SENTINEL).all()), "lse past total_tokens was written"
    # a sequence whose offsets are valid is computed as usual
    b, n = good
    b0, b1 = cu[b], cu[b + 1]
    o_ref, l_ref = oracle.prefill(c.q[b0:b1], c.k[b0:b1], c.v[b0:b1], c.sink, [0, b1 - b0],
                                  window=window, rope_base=base, scale=c.scale)
    compare(out_full[b0:b0 + n], lse_full[b0:b0 + n], o_ref[:n], l_ref[:n],
            f"valid sequence of {cu}")
    # the context still works and the status word was cleared
    out2, _ = ha.prefill(q, k, v, sink, torch.tensor([0, total], dtype=torch.int32, device=dev),
                         max_seqlen=total, window=window, rope_base=base)
    torch.cuda.synchronize()
    assert ha.hattn_check_device_status() == ha.HATTN_OK


@pytest.mark.parametrize("window,base", [(128, 1e4), (0, 5e6)])
def test_backward_skips_and_reports_bad_offsets(window, base):
    dev = torch.device("cuda")
    total, G = 300, 8
    c = synth.prefill_case([total], 2 * G, 2, window=window, rope_base=base, seed=902)
    q, k, v, sink = c.q.to(dev), c.k.to(dev), c.v.to(dev), c.sink.to(dev)
    cu = [0, 100, 400]  # the second sequence runs past total_tokens
    cu_d = torch.tensor(cu, dtype=torch.int32, device=dev)
    out = torch.zeros((total, c.hq, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((total, c.hq), dtype=torch.float32, device=dev)
    ha.prefill(q, k, v, sink, cu_d, max_seqlen=total, window=window, rope_base=base, out=out,
               lse=lse)
    torch.cuda.synchronize()
    assert ha.hattn_check_device_status() == ha.HATTN_ERR_INVALID_ARG
    dout = synth.randn_bf16((total, c.hq, 128), synth._gen(903, "cpu"), "cpu")
    dq = _slack(tuple(q.shape), torch.bfloat16, dev)
    dk = _slack(tuple(k.shape), torch.bfloat16, dev)
    dv = _slack(tuple(v.shape), torch.bfloat16, dev)
    ds = torch.empty((c.hq,), dtype=torch.float32, device=dev)
    ws = torch.empty(ha.hattn_prefill_backward_workspace_size(total, c.hq, c.hkv),
                     dtype=torch.uint8, device=dev)
    st = ha.hattn_prefill_backward(q, k, v, sink, out, lse, dout.to(dev), dq, dk, dv, ds, 2, cu_d,
                                   total, total, c.hq, c.hkv, 192, 128, 64, base, window, c.scale,
                                   ws, ws.numel())
    assert st == ha.HATTN_OK
    torch.cuda.synchronize()
    assert ha.hattn_check_device_status() == ha.HATTN_ERR_INVALID_ARG
    for name, t, n in (("dq", dq, total), ("dk", dk, total), ("dv", dv, total)):
        assert bool((t[n:] == SENTINEL).all()), f"{name} rows past total_tokens were written"
    # the valid first sequence's gradients match the oracle
    ref = oracle.prefill_backward(c.q[:100], c.k[:100], c.v[:100], c.sink, dout[:100], [0, 100],
                                  window=window, rope_base=base, scale=c.scale)
    for name, a, b in zip(("dq", "dk", "dv"), (dq[:100], dk[:100], dv[:100]), ref[:3]):
        a = a.double().cpu().numpy()
        rel = float(np.linalg.norm(a - b) / np.linalg.norm(b))
        assert rel < 1e-2, (name, rel)


def test_prefill_cached_skips_and_reports_prefix_past_the_cache():
    dev = torch.device("cuda")
    G, hkv, window, base = 8, 2, 0, 5e6
    hq = G * hkv
    prefixes, news, cap = [10, 50], [20, 30], 64  # 50 + 30 > 64
    d = synth.decode_case([p + n for p, n in zip(prefixes, news)], 1, hq, hkv, window=window,
                          rope_base=base, seed=904)
    kc = torch.zeros((2, hkv, cap, 192), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros((2, hkv, cap, 128), dtype=torch.bfloat16, device=dev)
    for b, P in enumerate(prefixes):
        ha.rope_kv_append(d.k_hist[b:b + 1, :P].contiguous().to(dev),
                          d.v_hist[b:b + 1, :P].contiguous().to(dev),
                          torch.zeros(1, dtype=torch.int32, device=dev), kc[b:b + 1],
                          vc[b:b + 1], is_ring=False, rope_base=base)
    g = synth._gen(905, "cpu")
    q_new = [synth.randn_bf16((n, hq, 192), g, "cpu") for n in news]
    k_new = torch.cat([d.k_hist[b, P:P + n] for b, (P, n) in enumerate(zip(prefixes, news))])
    v_new = torch.cat([d.v_hist[b, P:P + n] for b, (P, n) in enumerate(zip(prefixes, news))])
    total = sum(news)
    out_full = _slack((total, hq, 128), torch.bfloat16, dev)
    lse_full = _slack((total, hq), torch.float32, dev)
    cu = torch.tensor([0, news[0], total], dtype=torch.int32, device=dev)
    pre = torch.tensor(prefixes, dtype=torch.int32, device=dev)
    ha.prefill_cached(torch.cat(q_new).to(dev), k_new.to(dev), v_new.to(dev), kc, vc, cu, pre,
                      d.sink.to(dev), max_seqlen=max(news), max_prefix=max(prefixes),
                      window=window, rope_base=base, softmax_scale=d.scale,
                      out=out_full[:total], lse=lse_full[:total])
    torch.cuda.synchronize()
    assert ha.hattn_check_device_status() == ha.HATTN_ERR_INVALID_ARG
    assert bool((out_full[total:] == SENTINEL).all())
    assert bool((lse_full[total:] == SENTINEL).all())
    # the rows of the sequence that runs past the cache are not written
    assert bool((out_full[news[0]:total] == SENTINEL).all())
    o, l = oracle.decode(q_new[0][None], d.k_hist[0:1], d.v_hist[0:1], [prefixes[0] + news[0]],
                         d.sink, window=window, rope_base=base, scale=d.scale)
    compare(out_full[:news[0]], lse_full[:news[0]], o[0], l[0], "valid cached sequence")


# (G, window, base): one-block window units (G = 8 and 16 at W = 128), a
# window whose band needs several key blocks (G = 4) and a global layer
@pytest.mark.parametrize("G,window,base", [(8, 128, 1e4), (16, 128, 1e4), (4, 128, 1e4),
                                           (8, 0, 5e6)])
def test_prefill_reports_rotated_keys_past_fp16(G, window, base):
    """Rotated key dims are stored as fp16; a key whose rotation leaves the
    fp16 range is reported as HATTN_ERR_INVALID_ARG.  x = y = 6e4 in the
    pair (0, 32): the rotated values reach 6e4 * sqrt(2) at positions whose
    angle (pos radians for frequency 0) is near pi/4 + k pi/2."""
    dev = torch.device("cuda")
    total = 300
    c = synth.prefill_case([total], 2 * G, 2, window=window, rope_base=base, seed=907)
    q, v, sink = c.q.to(dev), c.v.to(dev), c.sink.to(dev)
    cu = c.cu_seqlens.to(dev)
    k_big = c.k.clone()
    k_big[:, :, 0] = 6e4
    k_big[:, :, 32] = 6e4
    ha.prefill(q, k_big.to(dev), v, sink, cu, max_seqlen=total, window=window, rope_base=base)
    torch.cuda.synchronize()
    assert ha.hattn_check_device_status() == ha.HATTN_ERR_INVALID_ARG
    # keys within range: no report, and the result matches the oracle
    out, lse = ha.prefill(q, c.k.to(dev), v, sink, cu, max_seqlen=total, window=window,
                          rope_base=base)
    torch.cuda.synchronize()
    assert ha.hattn_check_device_status() == ha.HATTN_OK
    o_ref, l_ref = oracle.prefill(c.q, c.k, c.v, c.sink, [0, total], window=window,
                                  rope_base=base, scale=c.scale)
    compare(out, lse, o_ref, l_ref, f"G {G} window {window}")
