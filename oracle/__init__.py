"""Plain fp64 CPU oracle for hybrid SWA / GA attention with a per-head sink.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this package.  The
product (``global_attention_sinks_gqa_b300``) never imports it, and the two
share no code: no kernels, headers, helpers, tables or constant generators.

Two independent implementations live here:

* ``hattn_oracle.c`` (loaded through ctypes): the definition written out row
  by row in double precision -- RoPE at each token's position, the visible key
  set, the logits, the softmax with the sink in its denominator, the weighted
  sum of values and the log-sum-exp -- and its backward (the chain rule
  through the same steps, for the gradients of q, k, v and the sink).
* ``brute.py`` (numpy): the same definition written as whole matrices (a sink
  column appended to an explicit masked logit matrix, RoPE as a complex
  rotation), forward and backward, used only on tiny shapes to cross-check the
  C oracle; its backward is pinned by finite differences of its forward.

Citations (page title, section): MiMo-V2-Flash Technical Report paper review
(xllm-io), sections 3.1 (shapes, GQA, partial RoPE, W = 128), 3.2 (learnable
sink in the softmax denominator) and 4 (RoPE bases 10K / 5M); plmsmile notes on
the MiMo series, MiMo-V2-Flash "local window" and "Learnable Attention Sink".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hattn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_hattn.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (-O2, OpenMP) next to its source."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall", "-Wextra",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i, l, d = ctypes.c_int, ctypes.c_long, ctypes.c_double
            lib.hattn_oracle_prefill.argtypes = [P, P, P, P, P, P, i, P, i, i, i, i, i, d, i, d,
                                                 P, l, i]
            lib.hattn_oracle_prefill.restype = i
            lib.hattn_oracle_decode.argtypes = [P, P, P, P, P, P, P, i, i, l, i, i, i, i, i, d,
                                                i, d, l, l, i, i]
            lib.hattn_oracle_decode.restype = i
            lib.hattn_oracle_rope.argtypes = [P, P, P, l, i, i, d]
            lib.hattn_oracle_rope.restype = i
            lib.hattn_oracle_prefill_backward.argtypes = [P, P, P, P, P, P, P, P, P, i, P, i, i, i,
                                                          i, i, d, i, d, i]
            lib.hattn_oracle_prefill_backward.restype = i
            lib.hattn_oracle_num_threads.argtypes = [i]
            lib.hattn_oracle_num_threads.restype = i
            _lib = lib
    return _lib


def _bf16_bits(x) -> np.ndarray:
    """bf16 tensor / uint16 array -> contiguous uint16 bit patterns."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            assert x.dtype == torch.bfloat16, x.dtype
            return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(x)
    assert a.dtype == np.uint16, a.dtype
    return a


def _f64(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().double().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads(nthreads: int = 0) -> int:
    """OpenMP threads the oracle uses for ``nthreads`` (0 = all cores)."""
    return _load().hattn_oracle_num_threads(nthreads)


def prefill(q, k, v, sink, cu_seqlens, *, window: int, rope_base: float, scale: float,
            rope_dim: int = 64, rows=None, nthreads: int = 0):
    """Prefill attention over packed sequences (positions restart at 0 per sequence).

    q [total, hq, dqk], k [total, hkv, dqk], v [total, hkv, dv] bf16 (un-rotated);
    sink [hq]; cu_seqlens [batch+1].  ``rows`` selects packed token indices.
    Returns (out [n_rows, hq, dv], lse [n_rows, hq]) as float64 arrays.
    """
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    total, hq, dqk = qb.shape
    hkv, dv = kb.shape[1], vb.shape[2]
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32).reshape(-1))
    assert cu[-1] == total and kb.shape[0] == total and vb.shape[0] == total
    s = _f64(sink).reshape(-1)
    assert s.shape[0] == hq
    if rows is None:
        n_rows, rows_p, rows_a = total, None, None
    else:
        rows_a = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        n_rows, rows_p = rows_a.shape[0], _ptr(rows_a)
    out = np.empty((n_rows, hq, dv), np.float64)
    lse = np.empty((n_rows, hq), np.float64)
    rc = _load().hattn_oracle_prefill(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(s), _ptr(out), _ptr(lse),
                                      len(cu) - 1, _ptr(cu), hq, hkv, dqk, dv, rope_dim,
                                      float(rope_base), int(window), float(scale), rows_p, n_rows,
                                      nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle prefill failed with code {rc}")
    return out, lse


def decode(q, k_hist, v_hist, seqlens, sink, *, window: int, rope_base: float, scale: float,
           rope_dim: int = 64, key_lo: int = 0, key_hi: int = -1, sink_on: bool = True,
           nthreads: int = 0):
    """Decode / MTP-verify: the last T tokens of each sequence over its history.

    q [B, T, hq, dqk] (un-rotated), k_hist [B, Lmax, hkv, dqk] (un-rotated, by
    absolute position), v_hist [B, Lmax, hkv, dv], seqlens [B] (>= T).
    Returns (out [B, T, hq, dv], lse [B, T, hq]) as float64 arrays.
    """
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k_hist), _bf16_bits(v_hist)
    B, T, hq, dqk = qb.shape
    Lmax, hkv = kb.shape[1], kb.shape[2]
    dv = vb.shape[3]
    sl = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32).reshape(-1))
    assert sl.shape[0] == B
    s = _f64(sink).reshape(-1)
    out = np.empty((B, T, hq, dv), np.float64)
    lse = np.empty((B, T, hq), np.float64)
    rc = _load().hattn_oracle_decode(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(sl), _ptr(s), _ptr(out),
                                     _ptr(lse), B, T, Lmax, hq, hkv, dqk, dv, rope_dim,
                                     float(rope_base), int(window), float(scale), int(key_lo),
                                     int(key_hi), 1 if sink_on else 0, nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle decode failed with code {rc}")
    return out, lse


def rope(x, positions, *, rope_base: float, rope_dim: int = 64):
    """RoPE of rows x [n, dim] (bf16) at integer positions [n]; float64 result."""
    xb = _bf16_bits(x)
    n, dim = xb.shape
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64).reshape(-1))
    assert pos.shape[0] == n
    y = np.empty((n, dim), np.float64)
    rc = _load().hattn_oracle_rope(_ptr(xb), _ptr(pos), _ptr(y), n, dim, rope_dim,
                                   float(rope_base))
    if rc != 0:
        raise RuntimeError(f"oracle rope failed with code {rc}")
    return y


def prefill_backward(q, k, v, sink, dout, cu_seqlens, *, window: int, rope_base: float,
                     scale: float, rope_dim: int = 64, nthreads: int = 0):
    """Gradients of sum(dout * out) of :func:`prefill` with respect to q, k, v
    (un-rotated inputs) and the sink logits.

    q, k, v as for :func:`prefill`; dout [total, hq, dv] bf16.  Returns
    (dq [total, hq, dqk], dk [total, hkv, dqk], dv [total, hkv, dv], dsink [hq])
    as float64 arrays.
    """
    qb, kb, vb, gb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v), _bf16_bits(dout)
    total, hq, dqk = qb.shape
    hkv, dv = kb.shape[1], vb.shape[2]
    assert gb.shape == (total, hq, dv)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32).reshape(-1))
    assert cu[-1] == total and kb.shape[0] == total and vb.shape[0] == total
    s = _f64(sink).reshape(-1)
    assert s.shape[0] == hq
    dq = np.empty((total, hq, dqk), np.float64)
    dk = np.empty((total, hkv, dqk), np.float64)
    dvv = np.empty((total, hkv, dv), np.float64)
    ds = np.empty((hq,), np.float64)
    rc = _load().hattn_oracle_prefill_backward(
        _ptr(qb), _ptr(kb), _ptr(vb), _ptr(s), _ptr(gb), _ptr(dq), _ptr(dk), _ptr(dvv), _ptr(ds),
        len(cu) - 1, _ptr(cu), hq, hkv, dqk, dv, rope_dim, float(rope_base), int(window),
        float(scale), nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle prefill backward failed with code {rc}")
    return dq, dk, dvv, ds
