"""Helpers for the GPU parity tests: run the CUDA path, compare with the oracle.

Tolerances (fp32 accumulation, bf16 inputs and outputs): max-abs <= 2e-2,
relative L2 <= 5e-3 over the compared set, |lse - lse_ref| <= 1e-3.
"""
import numpy as np
import torch

import global_attention_sinks_gqa_b300 as ha
import oracle
import synth

TOL_MAXABS = 2e-2
TOL_RELL2 = 5e-3
TOL_LSE = 1e-3


def compare(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    o = out_gpu.detach().float().cpu().double().numpy().reshape(out_ref.shape)
    l = lse_gpu.detach().cpu().double().numpy().reshape(lse_ref.shape)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    assert np.isfinite(l).all(), f"{what}: non-finite lse"
    maxabs = float(np.abs(o - out_ref).max())
    rel = float(np.linalg.norm(o - out_ref) / max(np.linalg.norm(out_ref), 1e-30))
    lerr = float(np.abs(l - lse_ref).max())
    msg = f"{what}: maxabs {maxabs:.3e} relL2 {rel:.3e} lse {lerr:.3e}"
    assert maxabs <= TOL_MAXABS, msg
    assert rel <= TOL_RELL2, msg
    assert lerr <= TOL_LSE, msg
    return dict(maxabs=maxabs, rel_l2=rel, lse_err=lerr)


def gpu_prefill(c: synth.PrefillCase):
    dev = torch.device("cuda")
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    sink, cu = c.sink.to(dev), c.cu_seqlens.to(dev)
    out, lse = ha.prefill(q, k, v, sink, cu, max_seqlen=c.max_seqlen, window=c.window,
                          rope_base=c.rope_base, softmax_scale=c.scale)
    torch.cuda.synchronize()
    ha.check_device_status()
    return out, lse


def oracle_prefill(c: synth.PrefillCase, rows=None, window=None):
    return oracle.prefill(c.q, c.k, c.v, c.sink, c.cu_seqlens.cpu().tolist(),
                          window=c.window if window is None else window, rope_base=c.rope_base,
                          scale=c.scale, rows=rows)


def fill_cache(d: synth.DecodeCase, cap: int, is_ring: bool, upto=None, init: float = 0.0):
    """KV caches holding positions [0, upto_b) of every sequence, written by
    the CUDA append kernel from the un-rotated history (ring: only the last
    cap positions, which are the ones a ring keeps).  Slots never written
    hold `init`."""
    dev = torch.device("cuda")
    B, hkv = d.B, d.hkv
    kc = torch.full((B, hkv, cap, synth.D_QK), init, dtype=torch.bfloat16, device=dev)
    vc = torch.full((B, hkv, cap, synth.D_V), init, dtype=torch.bfloat16, device=dev)
    kh = d.k_hist if d.k_hist.is_cuda else d.k_hist.to(dev)
    vh = d.v_hist if d.v_hist.is_cuda else d.v_hist.to(dev)
    for b in range(B):
        L = d.seqlens[b] if upto is None else upto[b]
        s = max(0, L - cap) if is_ring else 0
        if L - s <= 0:
            continue
        pos = torch.tensor([s], dtype=torch.int32, device=dev)
        ha.rope_kv_append(kh[b:b + 1, s:L].contiguous(), vh[b:b + 1, s:L].contiguous(), pos,
                          kc[b:b + 1], vc[b:b + 1], is_ring=is_ring, rope_base=d.rope_base)
    return kc, vc
