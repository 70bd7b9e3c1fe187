"""Hybrid sliding-window / global GQA attention with a learnable sink, on B300.

The compute lives in ``libhattn.so`` (hand-written sm_103a CUDA behind the C
ABI of ``include/hattn.h``).  This package is its Python binding:

* ``hattn_prefill``, ``hattn_rope_kv_append``, ``hattn_decode``, ... -- the C
  entry points under the same names, arguments marshalled with ctypes
  (tensors become their device pointers); they return the status code.
* ``prefill``, ``rope_kv_append``, ``decode`` -- conveniences that take torch
  CUDA tensors, allocate the outputs and the workspace with torch, call the C
  entry point on torch's current stream and raise on a non-zero status.

There is no fallback: if the library is missing or fails to load, every call
raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhattn.so")

HATTN_OK = 0
HATTN_ERR_INVALID_ARG = 1
HATTN_ERR_UNSUPPORTED = 2
HATTN_ERR_CUDA = 3
HATTN_ERR_RING_TOO_SMALL = 4
HATTN_ERR_TIMEOUT = 5
HATTN_ERR_WORKSPACE = 6

D_QK, D_V, ROPE_DIM = 192, 128, 64

# name -> (restype, argtypes)
_P, _I, _L, _F, _Z = (ctypes.c_void_p, ctypes.c_int, ctypes.c_long, ctypes.c_float,
                      ctypes.c_size_t)
SIGNATURES = {
    "hattn_version": (_I, []),
    "hattn_status_string": (ctypes.c_char_p, [_I]),
    "hattn_prefill_workspace_size": (_Z, [_L, _I, _I]),
    "hattn_prefill": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _L, _I, _I, _I, _I, _I, _I, _F, _I, _F,
                           _P, _Z, _P]),
    "hattn_prefill_cached": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _L, _I, _I, _I, _I,
                                  _I, _I, _I, _I, _F, _I, _F, _P, _Z, _P]),
    "hattn_prefill_shard": (_I, [_P, _P, _P, _P, _P, _P, _L, _I, _L, _I, _I, _I, _I, _I, _F, _I,
                                 _F, _P, _Z, _P]),
    "hattn_prefill_backward_workspace_size": (_Z, [_L, _I, _I]),
    "hattn_prefill_backward": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _L, _I, _I,
                                    _I, _I, _I, _I, _F, _I, _F, _P, _Z, _P]),
    "hattn_rope_kv_append": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "hattn_decode_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I, _I, _I, _I]),
    "hattn_decode": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                          _F, _F, _P, _Z, _P]),
    "hattn_decode_append": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                 _I, _I, _I, _I, _F, _F, _P, _Z, _P]),
    "hattn_decode_append_paged": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _I, _I,
                                       _I, _I, _I, _I, _I, _I, _I, _F, _F, _P, _Z, _P]),
    "hattn_decode_static_scratch": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                         _I, _I, _I, _I, _F, _F, _P]),
    "hattn_check_device_status": (_I, [_P]),
    "hattn_set_wait_limit_ns": (_I, [ctypes.c_ulonglong]),
    "hattn_selftest_lost_arrival": (_I, [_P]),
    "hattn_test_fail_next_launches": (_I, [_I]),
}

_lib = None


class HattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what} failed: {status_string(status)} ({status})")


def load_library(path: str = LIB_PATH):
    """Load libhattn.so (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"libhattn.so not found at {path}; build it with "
                               "`python -m global_attention_sinks_gqa_b300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.data_ptr() if x.numel() else None
    return int(x)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


# ---------------------------------------------------------------- C names
def hattn_version() -> int:
    return load_library().hattn_version()


def status_string(status: int) -> str:
    return load_library().hattn_status_string(int(status)).decode()


hattn_status_string = status_string


def hattn_prefill_workspace_size(total_tokens, hkv, dqk=D_QK) -> int:
    return load_library().hattn_prefill_workspace_size(int(total_tokens), int(hkv), int(dqk))


def hattn_prefill_backward_workspace_size(total_tokens, hq, hkv) -> int:
    return load_library().hattn_prefill_backward_workspace_size(int(total_tokens), int(hq),
                                                                int(hkv))


def hattn_prefill_backward(q, k, v, sink, out, lse, dout, grad_q, grad_k, grad_v, grad_sink, batch,
                           cu_seqlens, total_tokens, max_seqlen, hq, hkv, dqk, dv, rope_dim,
                           rope_base, window, softmax_scale, workspace, workspace_bytes,
                           stream=None) -> int:
    return load_library().hattn_prefill_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(sink), _ptr(out), _ptr(lse), _ptr(dout), _ptr(grad_q),
        _ptr(grad_k), _ptr(grad_v), _ptr(grad_sink), int(batch), _ptr(cu_seqlens),
        int(total_tokens), int(max_seqlen), int(hq), int(hkv), int(dqk), int(dv), int(rope_dim),
        float(rope_base), int(window), float(softmax_scale), _ptr(workspace),
        int(workspace_bytes), _stream(stream))


def hattn_prefill(q, k, v, sink, out, lse, batch, cu_seqlens, total_tokens, max_seqlen, hq, hkv,
                  dqk, dv, rope_dim, rope_base, window, softmax_scale, workspace, workspace_bytes,
                  stream=None) -> int:
    return load_library().hattn_prefill(
        _ptr(q), _ptr(k), _ptr(v), _ptr(sink), _ptr(out), _ptr(lse), int(batch), _ptr(cu_seqlens),
        int(total_tokens), int(max_seqlen), int(hq), int(hkv), int(dqk), int(dv), int(rope_dim),
        float(rope_base), int(window), float(softmax_scale), _ptr(workspace), int(workspace_bytes),
        _stream(stream))


def hattn_prefill_shard(q, k, v, sink, out, lse, shard_tokens, halo, pos0, hq, hkv, dqk, dv,
                        rope_dim, rope_base, window, softmax_scale, workspace, workspace_bytes,
                        stream=None) -> int:
    return load_library().hattn_prefill_shard(
        _ptr(q), _ptr(k), _ptr(v), _ptr(sink), _ptr(out), _ptr(lse), int(shard_tokens), int(halo),
        int(pos0), int(hq), int(hkv), int(dqk), int(dv), int(rope_dim), float(rope_base),
        int(window), float(softmax_scale), _ptr(workspace), int(workspace_bytes), _stream(stream))


def hattn_prefill_cached(q, k_new, v_new, k_cache, v_cache, cu_seqlens, prefix_lens, sink, out,
                         lse, batch, total_tokens, max_seqlen, max_prefix, cap, hq, hkv, dqk, dv,
                         rope_dim, rope_base, window, softmax_scale, workspace, workspace_bytes,
                         stream=None) -> int:
    return load_library().hattn_prefill_cached(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(cu_seqlens),
        _ptr(prefix_lens), _ptr(sink), _ptr(out), _ptr(lse), int(batch), int(total_tokens),
        int(max_seqlen), int(max_prefix), int(cap), int(hq), int(hkv), int(dqk), int(dv),
        int(rope_dim), float(rope_base), int(window), float(softmax_scale), _ptr(workspace),
        int(workspace_bytes), _stream(stream))


def hattn_rope_kv_append(k_new, v_new, start_pos, k_cache, v_cache, B, T, hkv, dqk, dv, cap,
                         is_ring, rope_dim, rope_base, stream=None) -> int:
    return load_library().hattn_rope_kv_append(
        _ptr(k_new), _ptr(v_new), _ptr(start_pos), _ptr(k_cache), _ptr(v_cache), int(B), int(T),
        int(hkv), int(dqk), int(dv), int(cap), int(is_ring), int(rope_dim), float(rope_base),
        _stream(stream))


def hattn_decode_workspace_size(B, T, hq, hkv, dv, max_seqlen_k, window, cap, is_ring) -> int:
    return load_library().hattn_decode_workspace_size(int(B), int(T), int(hq), int(hkv), int(dv),
                                                      int(max_seqlen_k), int(window), int(cap),
                                                      int(is_ring))


def hattn_decode(q, k_cache, v_cache, seqlens_k, sink, out, lse, B, T, hq, hkv, dqk, dv, cap,
                 is_ring, window, max_seqlen_k, rope_dim, rope_base, softmax_scale, workspace,
                 workspace_bytes, stream=None) -> int:
    return load_library().hattn_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens_k), _ptr(sink), _ptr(out), _ptr(lse),
        int(B), int(T), int(hq), int(hkv), int(dqk), int(dv), int(cap), int(is_ring), int(window),
        int(max_seqlen_k), int(rope_dim), float(rope_base), float(softmax_scale), _ptr(workspace),
        int(workspace_bytes), _stream(stream))


def hattn_decode_append(q, k_new, v_new, k_cache, v_cache, seqlens_k, sink, out, lse, B, T, hq,
                        hkv, dqk, dv, cap, is_ring, window, max_seqlen_k, rope_dim, rope_base,
                        softmax_scale, workspace, workspace_bytes, stream=None) -> int:
    return load_library().hattn_decode_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens_k),
        _ptr(sink), _ptr(out), _ptr(lse), int(B), int(T), int(hq), int(hkv), int(dqk), int(dv),
        int(cap), int(is_ring), int(window), int(max_seqlen_k), int(rope_dim), float(rope_base),
        float(softmax_scale), _ptr(workspace), int(workspace_bytes), _stream(stream))


def hattn_decode_append_paged(q, k_new, v_new, k_pages, v_pages, block_table, table_stride,
                              num_pages, page, seqlens_k, sink, out, lse, B, T, hq, hkv, dqk, dv,
                              window, max_seqlen_k, rope_dim, rope_base, softmax_scale,
                              workspace, workspace_bytes, stream=None) -> int:
    return load_library().hattn_decode_append_paged(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
        int(table_stride), int(num_pages), int(page), _ptr(seqlens_k), _ptr(sink), _ptr(out),
        _ptr(lse), int(B), int(T), int(hq), int(hkv), int(dqk), int(dv), int(window),
        int(max_seqlen_k), int(rope_dim), float(rope_base), float(softmax_scale), _ptr(workspace),
        int(workspace_bytes), _stream(stream))


def hattn_decode_static_scratch(q, k_cache, v_cache, seqlens_k, sink, out, lse, B, T, hq, hkv,
                                dqk, dv, cap, is_ring, window, max_seqlen_k, rope_dim, rope_base,
                                softmax_scale, stream=None) -> int:
    """hattn_decode() without a caller workspace, for callers that cannot
    allocate device memory: the library's fixed scratch array is used instead
    (see include/hattn.h for its size and sharing rules)."""
    return load_library().hattn_decode_static_scratch(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens_k), _ptr(sink), _ptr(out), _ptr(lse),
        int(B), int(T), int(hq), int(hkv), int(dqk), int(dv), int(cap), int(is_ring), int(window),
        int(max_seqlen_k), int(rope_dim), float(rope_base), float(softmax_scale), _stream(stream))


def hattn_check_device_status(stream=None) -> int:
    return load_library().hattn_check_device_status(_stream(stream))


def hattn_set_wait_limit_ns(limit_ns: int) -> int:
    return load_library().hattn_set_wait_limit_ns(int(limit_ns))


def hattn_selftest_lost_arrival(stream=None) -> int:
    return load_library().hattn_selftest_lost_arrival(_stream(stream))


def hattn_test_fail_next_launches(n: int) -> int:
    return load_library().hattn_test_fail_next_launches(int(n))


# ---------------------------------------------------------------- conveniences
def _check(status: int, what: str):
    if status != HATTN_OK:
        raise HattnError(status, what)


def prefill(q, k, v, sink, cu_seqlens, *, max_seqlen: int, window: int, rope_base: float,
            softmax_scale: float | None = None, out=None, lse=None, workspace=None,
            with_lse: bool = True):
    """One layer's prefill over packed sequences; returns (out, lse)."""
    total, hq, dqk = q.shape
    hkv, dv = k.shape[1], v.shape[2]
    if softmax_scale is None:
        softmax_scale = dqk ** -0.5
    if out is None:
        out = torch.empty((total, hq, dv), dtype=torch.bfloat16, device=q.device)
    if lse is None and with_lse:
        lse = torch.empty((total, hq), dtype=torch.float32, device=q.device)
    need = hattn_prefill_workspace_size(total, hkv, dqk)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(hattn_prefill(q, k, v, sink, out, lse, cu_seqlens.numel() - 1, cu_seqlens, total,
                         max_seqlen, hq, hkv, dqk, dv, ROPE_DIM, rope_base, window, softmax_scale,
                         workspace, workspace.numel()), "hattn_prefill")
    return out, lse


def prefill_shard(q, k, v, sink, *, pos0: int, halo: int, window: int, rope_base: float,
                  softmax_scale: float | None = None, out=None, lse=None, workspace=None,
                  with_lse: bool = True):
    """One context-parallel shard of a layer's prefill: q [L, hq, dqk] holds the
    shard's queries (positions pos0 .. pos0 + L - 1), k / v [halo + L, hkv, d]
    the halo's keys and values followed by the shard's own.  Returns (out, lse)."""
    L, hq, dqk = q.shape
    hkv, dv = k.shape[1], v.shape[2]
    assert k.shape[0] == halo + L and v.shape[0] == halo + L
    if softmax_scale is None:
        softmax_scale = dqk ** -0.5
    if out is None:
        out = torch.empty((L, hq, dv), dtype=torch.bfloat16, device=q.device)
    if lse is None and with_lse:
        lse = torch.empty((L, hq), dtype=torch.float32, device=q.device)
    need = hattn_prefill_workspace_size(halo + L, hkv, dqk)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(hattn_prefill_shard(q, k, v, sink, out, lse, L, halo, pos0, hq, hkv, dqk, dv, ROPE_DIM,
                               rope_base, window, softmax_scale, workspace, workspace.numel()),
           "hattn_prefill_shard")
    return out, lse


def prefill_backward(q, k, v, sink, out, lse, dout, cu_seqlens, *, max_seqlen: int, window: int,
                     rope_base: float, softmax_scale: float | None = None, workspace=None):
    """Gradients of one layer's prefill; returns (grad_q, grad_k, grad_v, grad_sink).
    out and lse are the forward's results for the same inputs."""
    total, hq, dqk = q.shape
    hkv, dv = k.shape[1], v.shape[2]
    if softmax_scale is None:
        softmax_scale = dqk ** -0.5
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dvv = torch.empty_like(v)
    ds = torch.empty((hq,), dtype=torch.float32, device=q.device)
    need = hattn_prefill_backward_workspace_size(total, hq, hkv)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(hattn_prefill_backward(q, k, v, sink, out, lse, dout, dq, dk, dvv, ds,
                                  cu_seqlens.numel() - 1, cu_seqlens, total, max_seqlen, hq, hkv,
                                  dqk, dv, ROPE_DIM, rope_base, window, softmax_scale, workspace,
                                  workspace.numel()), "hattn_prefill_backward")
    return dq, dk, dvv, ds


def prefill_cached(q, k_new, v_new, k_cache, v_cache, cu_seqlens, prefix_lens, sink, *,
                   max_seqlen: int, max_prefix: int, window: int, rope_base: float,
                   softmax_scale: float | None = None, out=None, lse=None, workspace=None,
                   with_lse: bool = True):
    """Prefill of new tokens that continue cached prefixes (linear caches); the new
    keys / values are appended to the caches.  Returns (out, lse)."""
    total, hq, dqk = q.shape
    hkv, dv = k_new.shape[1], v_new.shape[2]
    cap = k_cache.shape[2]
    if softmax_scale is None:
        softmax_scale = dqk ** -0.5
    if out is None:
        out = torch.empty((total, hq, dv), dtype=torch.bfloat16, device=q.device)
    if lse is None and with_lse:
        lse = torch.empty((total, hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(256, dtype=torch.uint8, device=q.device)
    _check(hattn_prefill_cached(q, k_new, v_new, k_cache, v_cache, cu_seqlens, prefix_lens, sink,
                                out, lse, cu_seqlens.numel() - 1, total, max_seqlen, max_prefix,
                                cap, hq, hkv, dqk, dv, ROPE_DIM, rope_base, window,
                                softmax_scale, workspace, workspace.numel()),
           "hattn_prefill_cached")
    return out, lse


def rope_kv_append(k_new, v_new, start_pos, k_cache, v_cache, *, is_ring: bool, rope_base: float):
    B, T, hkv, dqk = k_new.shape
    cap = k_cache.shape[2]
    _check(hattn_rope_kv_append(k_new, v_new, start_pos, k_cache, v_cache, B, T, hkv, dqk,
                                v_new.shape[3], cap, 1 if is_ring else 0, ROPE_DIM, rope_base),
           "hattn_rope_kv_append")


def decode(q, k_cache, v_cache, seqlens_k, sink, *, max_seqlen_k: int, window: int,
           is_ring: bool, rope_base: float, softmax_scale: float | None = None, out=None,
           lse=None, workspace=None, with_lse: bool = True):
    """Decode / verify step for T = q.shape[1] tokens per sequence; returns (out, lse)."""
    B, T, hq, dqk = q.shape
    hkv, cap = k_cache.shape[1], k_cache.shape[2]
    dv = v_cache.shape[3]
    if softmax_scale is None:
        softmax_scale = dqk ** -0.5
    if out is None:
        out = torch.empty((B, T, hq, dv), dtype=torch.bfloat16, device=q.device)
    if lse is None and with_lse:
        lse = torch.empty((B, T, hq), dtype=torch.float32, device=q.device)
    need = hattn_decode_workspace_size(B, T, hq, hkv, dv, max_seqlen_k, window, cap,
                                       1 if is_ring else 0)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(hattn_decode(q, k_cache, v_cache, seqlens_k, sink, out, lse, B, T, hq, hkv, dqk, dv,
                        cap, 1 if is_ring else 0, window, max_seqlen_k, ROPE_DIM, rope_base,
                        softmax_scale, workspace, workspace.numel() if workspace is not None else 0),
           "hattn_decode")
    return out, lse


def decode_append(q, k_new, v_new, k_cache, v_cache, seqlens_k, sink, *, max_seqlen_k: int,
                  window: int, is_ring: bool, rope_base: float,
                  softmax_scale: float | None = None, out=None, lse=None, workspace=None,
                  with_lse: bool = True):
    """Append the T = q.shape[1] new tokens' K/V to the caches and run the
    decode / verify step over them; returns (out, lse)."""
    B, T, hq, dqk = q.shape
    hkv, cap = k_cache.shape[1], k_cache.shape[2]
    dv = v_cache.shape[3]
    if softmax_scale is None:
        softmax_scale = dqk ** -0.5
    if out is None:
        out = torch.empty((B, T, hq, dv), dtype=torch.bfloat16, device=q.device)
    if lse is None and with_lse:
        lse = torch.empty((B, T, hq), dtype=torch.float32, device=q.device)
    need = hattn_decode_workspace_size(B, T, hq, hkv, dv, max_seqlen_k, window, cap,
                                       1 if is_ring else 0)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(hattn_decode_append(q, k_new, v_new, k_cache, v_cache, seqlens_k, sink, out, lse, B, T,
                               hq, hkv, dqk, dv, cap, 1 if is_ring else 0, window, max_seqlen_k,
                               ROPE_DIM, rope_base, softmax_scale, workspace,
                               workspace.numel() if workspace is not None else 0),
           "hattn_decode_append")
    return out, lse


def decode_append_paged(q, k_new, v_new, k_pages, v_pages, block_table, seqlens_k, sink, *,
                        max_seqlen_k: int, window: int, rope_base: float,
                        softmax_scale: float | None = None, out=None, lse=None, workspace=None,
                        with_lse: bool = True):
    """decode_append over paged caches k_pages / v_pages [num_pages, hkv, page, d] and
    block_table [B, table_stride] (int32); returns (out, lse)."""
    B, T, hq, dqk = q.shape
    num_pages, hkv, page, _ = k_pages.shape
    dv = v_pages.shape[3]
    stride = block_table.shape[1]
    if softmax_scale is None:
        softmax_scale = dqk ** -0.5
    if out is None:
        out = torch.empty((B, T, hq, dv), dtype=torch.bfloat16, device=q.device)
    if lse is None and with_lse:
        lse = torch.empty((B, T, hq), dtype=torch.float32, device=q.device)
    need = hattn_decode_workspace_size(B, T, hq, hkv, dv, max_seqlen_k, window, stride * page, 0)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(hattn_decode_append_paged(q, k_new, v_new, k_pages, v_pages, block_table, stride,
                                     num_pages, page, seqlens_k, sink, out, lse, B, T, hq, hkv,
                                     dqk, dv, window, max_seqlen_k, ROPE_DIM, rope_base,
                                     softmax_scale, workspace,
                                     workspace.numel() if workspace is not None else 0),
           "hattn_decode_append_paged")
    return out, lse


def check_device_status(stream=None):
    _check(hattn_check_device_status(stream), "device status")
