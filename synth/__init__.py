"""Seeded synthetic inputs for hybrid SWA / GA sink attention.

This module is shared by the tests, the bench and the oracle checks.  It holds
no attention arithmetic at all: only shapes, seeds and random draws, so that
the CUDA path and the CPU oracle see identical bf16 values without sharing any
of the method's code.

Recipe (the workloads of the MiMo-V2-Flash hybrid attention layer; shapes from
the MiMo-V2-Flash paper review, section 3.1, and the decode batch of 64 from
the plmsmile notes, "MTP decoding gains"):

* q, k, v ~ N(0, 1) drawn in fp32 and rounded to bf16 (round-to-nearest-even);
* sink ~ N(sink_mean, sink_std) in fp32, one per query head;
* draw order inside one case: q, k, v, sink; sequence lengths, when random,
  come from a second generator seeded with ``seed + 7919`` so that they never
  shift the tensor draws;
* a ``torch.Generator`` on the device the tensors are created on.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

D_QK = 192
D_V = 128
ROPE_DIM = 64
WINDOW = 128
SWA_BASE = 1.0e4
GA_BASE = 5.0e6


def default_scale(dqk: int = D_QK) -> float:
    return 1.0 / math.sqrt(dqk)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, gen: torch.Generator, device, mean: float = 0.0,
               std: float = 1.0) -> torch.Tensor:
    x = torch.randn(tuple(shape), generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(torch.bfloat16)


def randn_f32(shape, gen: torch.Generator, device, mean: float = 0.0,
              std: float = 1.0) -> torch.Tensor:
    x = torch.randn(tuple(shape), generator=gen, device=device, dtype=torch.float32)
    return x * std + mean


@dataclass
class PrefillCase:
    q: torch.Tensor          # bf16 [total, hq, dqk]
    k: torch.Tensor          # bf16 [total, hkv, dqk]
    v: torch.Tensor          # bf16 [total, hkv, dv]
    sink: torch.Tensor       # fp32 [hq]
    cu_seqlens: torch.Tensor  # int32 [batch + 1] (on the same device)
    seqlens: list
    hq: int
    hkv: int
    window: int
    rope_base: float
    scale: float

    @property
    def total(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_seqlen(self) -> int:
        return max(self.seqlens)


def prefill_case(seqlens, hq: int, hkv: int, *, window: int, rope_base: float, seed: int,
                 device="cpu", dqk: int = D_QK, dv: int = D_V, sink_mean: float = 0.0,
                 sink_std: float = 1.0, scale: float | None = None) -> PrefillCase:
    seqlens = [int(s) for s in seqlens]
    total = sum(seqlens)
    g = _gen(seed, device)
    q = randn_bf16((total, hq, dqk), g, device)
    k = randn_bf16((total, hkv, dqk), g, device)
    v = randn_bf16((total, hkv, dv), g, device)
    sink = randn_f32((hq,), g, device, sink_mean, sink_std)
    cu = [0]
    for s in seqlens:
        cu.append(cu[-1] + s)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=device)
    return PrefillCase(q, k, v, sink, cu_t, seqlens, hq, hkv, window, rope_base,
                       default_scale(dqk) if scale is None else scale)


def random_lengths(n: int, lo: int, hi: int, seed: int) -> list:
    """n integer lengths uniform in [lo, hi] (inclusive), CPU generator."""
    g = _gen(seed + 7919, "cpu")
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


@dataclass
class DecodeCase:
    q: torch.Tensor          # bf16 [B, T, hq, dqk]   queries at positions L-T .. L-1
    k_hist: torch.Tensor     # bf16 [B, Lmax, hkv, dqk] un-rotated keys by position
    v_hist: torch.Tensor     # bf16 [B, Lmax, hkv, dv]
    sink: torch.Tensor       # fp32 [hq]
    seqlens: list            # L_b, tokens including the T new ones
    hq: int
    hkv: int
    window: int
    rope_base: float
    scale: float

    @property
    def B(self) -> int:
        return int(self.q.shape[0])

    @property
    def T(self) -> int:
        return int(self.q.shape[1])


def decode_case(seqlens, T: int, hq: int, hkv: int, *, window: int, rope_base: float, seed: int,
                device="cpu", lmax: int | None = None, dqk: int = D_QK, dv: int = D_V,
                sink_mean: float = 0.0, sink_std: float = 1.0,
                scale: float | None = None) -> DecodeCase:
    seqlens = [int(s) for s in seqlens]
    B = len(seqlens)
    Lmax = max(seqlens) if lmax is None else int(lmax)
    g = _gen(seed, device)
    q = randn_bf16((B, T, hq, dqk), g, device)
    k = randn_bf16((B, Lmax, hkv, dqk), g, device)
    v = randn_bf16((B, Lmax, hkv, dv), g, device)
    sink = randn_f32((hq,), g, device, sink_mean, sink_std)
    return DecodeCase(q, k, v, sink, seqlens, hq, hkv, window, rope_base,
                      default_scale(dqk) if scale is None else scale)


# The five workloads of the hybrid attention layer (sizes as stated for the
# MiMo-V2-Flash attention stack; seeds 0, 2, 3, 4, 5).
CONFIGS = {
    "tiny_swa": dict(kind="prefill", seqlens=[512], hq=8, hkv=1, window=WINDOW,
                     rope_base=SWA_BASE, seed=0),
    "swa_prefill_32k": dict(kind="prefill", seqlens=[32768], hq=64, hkv=8, window=WINDOW,
                            rope_base=SWA_BASE, seed=2),
    "ga_prefill_32k": dict(kind="prefill", seqlens=[32768], hq=64, hkv=4, window=0,
                           rope_base=GA_BASE, seed=3),
    "decode_b64_t4": dict(kind="decode", B=64, T=4, lens=(8192, 65536), seed=4,
                          swa=dict(hq=64, hkv=8, window=WINDOW, rope_base=SWA_BASE),
                          ga=dict(hq=64, hkv=4, window=0, rope_base=GA_BASE)),
    "hybrid_block_256k": dict(kind="hybrid", seqlens=[262144], seed=5, n_swa=5,
                              swa=dict(hq=64, hkv=8, window=WINDOW, rope_base=SWA_BASE),
                              ga=dict(hq=64, hkv=4, window=0, rope_base=GA_BASE)),
}
