"""Context parallelism for a layer's prefill: one sequence cut into consecutive
shards, one per rank, and the halo exchange that a shard needs before
``hattn_prefill_shard`` can run on it.

plmsmile notes on the MiMo series, MiMo-V2.6, "DFlash and long-context system
optimisation" (training memory): context parallelism of the sliding-window
layers exchanges only the keys and values the window can reach, never the
whole history.  A query at position p of a window layer sees keys
p - window + 1 .. p, so the shard that starts at pos0 needs the last
min(window - 1, pos0) keys and values before it -- its halo.  When the shards
are at least window - 1 tokens long the halo comes from the previous rank
alone; shorter shards take theirs from several earlier ranks.  A global layer
(window 0) needs the whole history as its halo (an all-gather of the earlier
shards), which the same bookkeeping describes.

Buffers: every rank keeps its keys and values in [halo + L, heads, dim]
buffers whose rows [halo, halo + L) hold its own shard (written there by
whatever produces them) and whose rows [0, halo) the exchange fills.  Halo
rows travel point to point, from the rank that owns them straight into the
receiver's own buffer (``torch.distributed`` send / receive: NCCL between
GPUs, gloo between CPU processes); no rank reads another's memory.

Nothing here computes attention: it is argument bookkeeping and data
movement around the C ABI.
"""
from __future__ import annotations

from typing import List, Tuple

import torch


def shard_bounds(seq_len: int, world: int, rank: int) -> Tuple[int, int]:
    """(pos0, length) of rank's shard: consecutive, near-equal shards, the
    first seq_len % world of them one token longer."""
    if world <= 0 or not 0 <= rank < world or seq_len < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(seq_len, world)
    pos0 = rank * base + min(rank, extra)
    return pos0, base + (1 if rank < extra else 0)


def halo_len(pos0: int, window: int) -> int:
    """Rows of keys before the shard that its queries can see."""
    if window < 0 or pos0 < 0:
        raise ValueError("bad halo request")
    return min(window - 1, pos0) if window > 0 else pos0


def halo_sources(seq_len: int, world: int, rank: int,
                 window: int) -> List[Tuple[int, int, int, int]]:
    """Where rank's halo comes from: (source rank, first row among the
    source's own rows, first row of the receiver's buffer, rows), in order of
    position; together they cover buffer rows [0, halo) once each."""
    pos0, _ = shard_bounds(seq_len, world, rank)
    h = halo_len(pos0, window)
    lo = pos0 - h  # first position the halo holds
    out = []
    for src in range(rank):
        s0, sl = shard_bounds(seq_len, world, src)
        a, b = max(s0, lo), min(s0 + sl, pos0)
        if a < b:
            out.append((src, a - s0, a - lo, b - a))
    return out


def halo_destinations(seq_len: int, world: int, rank: int,
                      window: int) -> List[Tuple[int, int, int, int]]:
    """What rank sends: (destination rank, first row among rank's own rows,
    first row of the destination's buffer, rows) -- the mirror of the
    destinations' halo_sources."""
    out = []
    for dst in range(rank + 1, world):
        for src, src_row, dst_row, n in halo_sources(seq_len, world, dst, window):
            if src == rank:
                out.append((dst, src_row, dst_row, n))
    return out


def exchange_halo(k_buf: torch.Tensor, v_buf: torch.Tensor, seq_len: int, window: int,
                  group=None) -> int:
    """Fill rows [0, halo) of this rank's k_buf / v_buf ([halo + L, heads, dim],
    rows [halo, halo + L) already holding the shard's own keys and values) with
    the halo, received from the ranks that own it; send this rank's rows that
    later ranks need.  Every rank of the group calls it.  Returns halo."""
    import torch.distributed as dist
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    pos0, length = shard_bounds(seq_len, world, rank)
    h = halo_len(pos0, window)
    if k_buf.shape[0] != h + length or v_buf.shape[0] != h + length:
        raise ValueError(f"rank {rank}: buffers need {h} + {length} rows")
    if not (k_buf.is_contiguous() and v_buf.is_contiguous()):
        raise ValueError("buffers must be contiguous")
    ops = []
    for dst, src_row, dst_row, n in halo_destinations(seq_len, world, rank, window):
        for buf in (k_buf, v_buf):
            ops.append(dist.P2POp(dist.isend, buf[h + src_row:h + src_row + n], dst, group))
    for src, src_row, dst_row, n in halo_sources(seq_len, world, rank, window):
        for buf in (k_buf, v_buf):
            ops.append(dist.P2POp(dist.irecv, buf[dst_row:dst_row + n], src, group))
    if ops:
        for req in dist.batch_isend_irecv(ops):
            req.wait()
    return h


def halo_from_shards(own: List[torch.Tensor], seq_len: int, window: int,
                     rank: int) -> torch.Tensor:
    """Single-process stand-in for the exchange: rank's [halo + L, ...] buffer
    assembled from every rank's own rows (own[r] = rank r's shard), following
    the same bookkeeping.  For running all shards of a sequence on one device."""
    world = len(own)
    pos0, length = shard_bounds(seq_len, world, rank)
    h = halo_len(pos0, window)
    mine = own[rank]
    if mine.shape[0] != length:
        raise ValueError("shard length mismatch")
    buf = torch.empty((h + length, *mine.shape[1:]), dtype=mine.dtype, device=mine.device)
    for src, src_row, dst_row, n in halo_sources(seq_len, world, rank, window):
        buf[dst_row:dst_row + n] = own[src][src_row:src_row + n]
    buf[h:] = mine
    return buf
