"""Brute-force numpy fp64 restatement of the attention definition (tiny shapes).

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).  It is written as whole
matrices so that it shares no structure with the row-by-row C oracle:

* RoPE as a complex rotation: dims (i, i + R/2) form z_i = x_i + 1j*x_{i+R/2},
  rotated by exp(1j * pos * theta_i), theta_i = base^(-2i/R) (MiMo-V2-Flash
  paper review, section 3.1: RoPE on the first 64 dims; section 4: bases).
* the logits of one head form an explicit [S, S] matrix, the invisible pairs
  are set to -inf (causal, and p - j < W for a window W > 0: plmsmile notes,
  MiMo-V2-Flash "local window"), and one extra column holding the sink logit
  is appended (paper review, section 3.2; plmsmile notes, "Learnable Attention
  Sink": the sink joins the denominator and has no value, i.e. a zero value
  row);
* softmax over the S + 1 columns, then out = P @ [V; 0] and lse = log-sum-exp
  of the row;
* backward (gradients of sum(dout * out)) in matrix form: dP = dout [V; 0]^T,
  dZ = P * (dP - rowsum(dP * P)) over all S + 1 columns (the sink's column
  gives the sink gradient), dQ' = scale dZ K', dK' = scale dZ^T Q',
  dV = P^T dout, and the rotation undone by the conjugate complex factor.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(x) -> np.ndarray:
    """bf16 torch tensor or uint16 bit array -> float64 (exact)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(x)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def rope_complex(x: np.ndarray, pos: np.ndarray, base: float, rope_dim: int) -> np.ndarray:
    """x [..., S, dim] rotated at positions pos [S] (complex-multiplication form)."""
    if rope_dim == 0:
        return x.copy()
    half = rope_dim // 2
    theta = base ** (-2.0 * np.arange(half) / rope_dim)
    rot = np.exp(1j * np.outer(pos.astype(np.float64), theta))  # [S, half]
    zc = x[..., :half] + 1j * x[..., half:rope_dim]
    zc = zc * rot
    y = x.copy()
    y[..., :half] = zc.real
    y[..., half:rope_dim] = zc.imag
    return y


def visible_mask(S_q: int, S_k: int, q_pos: np.ndarray, window: int) -> np.ndarray:
    """[S_q, S_k] boolean: key j visible to a query at q_pos[i]."""
    j = np.arange(S_k)[None, :]
    p = q_pos[:, None]
    m = j <= p
    if window > 0:
        m &= (p - j) < window
    return m


def attention_one_sequence(q, k, v, sink, *, window, rope_base, scale, rope_dim=64,
                           q_pos=None):
    """One sequence.  q [Sq, hq, dqk], k [Sk, hkv, dqk], v [Sk, hkv, dv] (float64,
    un-rotated); keys sit at positions 0..Sk-1, queries at q_pos (default
    0..Sq-1).  Returns out [Sq, hq, dv], lse [Sq, hq]."""
    Sq, hq, dqk = q.shape
    Sk, hkv, _ = k.shape
    dv = v.shape[2]
    G = hq // hkv
    if q_pos is None:
        q_pos = np.arange(Sq)
    qh = rope_complex(np.transpose(q, (1, 0, 2)), q_pos, rope_base, rope_dim)   # [hq, Sq, d]
    kh = rope_complex(np.transpose(k, (1, 0, 2)), np.arange(Sk), rope_base, rope_dim)
    vh = np.transpose(v, (1, 0, 2))                                            # [hkv, Sk, dv]
    mask = visible_mask(Sq, Sk, np.asarray(q_pos), window)
    out = np.zeros((Sq, hq, dv))
    lse = np.zeros((Sq, hq))
    for h in range(hq):
        g = h // G
        logits = scale * qh[h] @ kh[g].T                                         # [Sq, Sk]
        logits = np.where(mask, logits, -np.inf)
        full = np.concatenate([logits, np.full((Sq, 1), float(sink[h]))], axis=1)
        mx = full.max(axis=1, keepdims=True)
        e = np.exp(full - mx)
        Z = e.sum(axis=1, keepdims=True)
        P = e / Z
        vext = np.concatenate([vh[g], np.zeros((1, dv))], axis=0)                 # sink value 0
        out[:, h, :] = P @ vext
        lse[:, h] = (mx + np.log(Z))[:, 0]
    return out, lse


def prefill(q, k, v, sink, cu_seqlens, *, window, rope_base, scale, rope_dim=64):
    """Packed varlen prefill (float64 results), one sequence at a time."""
    qd, kd, vd = bf16_to_f64(q), bf16_to_f64(k), bf16_to_f64(v)
    sd = np.asarray(sink, dtype=np.float64).reshape(-1)
    cu = np.asarray(cu_seqlens).reshape(-1)
    outs, lses = [], []
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        o, l = attention_one_sequence(qd[a:e], kd[a:e], vd[a:e], sd, window=window,
                                      rope_base=rope_base, scale=scale, rope_dim=rope_dim)
        outs.append(o)
        lses.append(l)
    return np.concatenate(outs, 0), np.concatenate(lses, 0)


def rope_complex_transposed(g: np.ndarray, pos: np.ndarray, base: float,
                            rope_dim: int) -> np.ndarray:
    """Gradient through :func:`rope_complex`: multiply by the conjugate rotation."""
    if rope_dim == 0:
        return g.copy()
    half = rope_dim // 2
    theta = base ** (-2.0 * np.arange(half) / rope_dim)
    rot = np.exp(-1j * np.outer(pos.astype(np.float64), theta))
    zc = (g[..., :half] + 1j * g[..., half:rope_dim]) * rot
    y = g.copy()
    y[..., :half] = zc.real
    y[..., half:rope_dim] = zc.imag
    return y


def attention_backward_one_sequence(q, k, v, sink, dout, *, window, rope_base, scale,
                                    rope_dim=64):
    """Gradients of sum(dout * out) for one sequence (float64 arrays as in
    :func:`attention_one_sequence`; dout [S, hq, dv]).  Returns dq, dk, dv,
    dsink [hq]."""
    S, hq, dqk = q.shape
    hkv, dv = k.shape[1], v.shape[2]
    G = hq // hkv
    pos = np.arange(S)
    qh = rope_complex(np.transpose(q, (1, 0, 2)), pos, rope_base, rope_dim)
    kh = rope_complex(np.transpose(k, (1, 0, 2)), pos, rope_base, rope_dim)
    vh = np.transpose(v, (1, 0, 2))
    gh = np.transpose(dout, (1, 0, 2))
    mask = visible_mask(S, S, pos, window)
    dqr = np.zeros((hq, S, dqk))
    dkr = np.zeros((hkv, S, dqk))
    dvh = np.zeros((hkv, S, dv))
    dsink = np.zeros(hq)
    for h in range(hq):
        g = h // G
        logits = np.where(mask, scale * qh[h] @ kh[g].T, -np.inf)
        full = np.concatenate([logits, np.full((S, 1), float(sink[h]))], axis=1)
        e = np.exp(full - full.max(axis=1, keepdims=True))
        P = e / e.sum(axis=1, keepdims=True)                       # [S, S + 1]
        vext = np.concatenate([vh[g], np.zeros((1, dv))], axis=0)
        dP = gh[h] @ vext.T                                        # [S, S + 1]
        dZ = P * (dP - (dP * P).sum(axis=1, keepdims=True))
        dsink[h] = dZ[:, S].sum()
        dZk = dZ[:, :S]
        dqr[h] = scale * dZk @ kh[g]
        dkr[g] += scale * dZk.T @ qh[h]
        dvh[g] += P[:, :S].T @ gh[h]
    dq = np.transpose(rope_complex_transposed(dqr, pos, rope_base, rope_dim), (1, 0, 2))
    dk = np.transpose(rope_complex_transposed(dkr, pos, rope_base, rope_dim), (1, 0, 2))
    return dq, dk, np.transpose(dvh, (1, 0, 2)), dsink


def prefill_backward(q, k, v, sink, dout, cu_seqlens, *, window, rope_base, scale, rope_dim=64):
    """Packed varlen backward (float64 results), one sequence at a time."""
    qd, kd, vd, gd = bf16_to_f64(q), bf16_to_f64(k), bf16_to_f64(v), bf16_to_f64(dout)
    sd = np.asarray(sink, dtype=np.float64).reshape(-1)
    cu = np.asarray(cu_seqlens).reshape(-1)
    dqs, dks, dvs = [], [], []
    dsink = np.zeros(sd.shape[0])
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        dq, dk, dv, ds = attention_backward_one_sequence(
            qd[a:e], kd[a:e], vd[a:e], sd, gd[a:e], window=window, rope_base=rope_base,
            scale=scale, rope_dim=rope_dim)
        dqs.append(dq)
        dks.append(dk)
        dvs.append(dv)
        dsink += ds
    return np.concatenate(dqs, 0), np.concatenate(dks, 0), np.concatenate(dvs, 0), dsink
