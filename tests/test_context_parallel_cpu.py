"""Context-parallel bookkeeping and the halo exchange, on CPU.

The shards of a sequence are consecutive and cover it once; a shard's halo
(min(window - 1, pos0) rows before it, or the whole history for a global
layer) is assembled from the owners' rows exactly once, and what each rank
sends is the mirror of what the others receive.  The exchange itself runs
with two and three gloo ranks (127.0.0.1), including shards shorter than the
halo, so that a halo spans several earlier ranks.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from global_attention_sinks_gqa_b300 import context_parallel as cp

CASES = [(1000, 2, 128), (1000, 3, 128), (300, 3, 128), (300, 4, 128), (257, 5, 1), (257, 5, 2),
         (500, 4, 0), (7, 4, 128), (4096, 8, 128), (3, 5, 128)]


@pytest.mark.parametrize("seq_len,world,window", CASES)
def test_shards_cover_the_sequence_and_halos_cover_the_window(seq_len, world, window):
    ends = 0
    for r in range(world):
        pos0, length = cp.shard_bounds(seq_len, world, r)
        assert pos0 == ends and length >= 0
        ends = pos0 + length
        h = cp.halo_len(pos0, window)
        assert h == (min(window - 1, pos0) if window else pos0)
        # the halo's rows, in order, each exactly once, from earlier shards
        covered = []
        for src, src_row, dst_row, n in cp.halo_sources(seq_len, world, r, window):
            s0, sl = cp.shard_bounds(seq_len, world, src)
            assert src < r and 0 <= src_row and src_row + n <= sl and n > 0
            covered += [(dst_row + i, s0 + src_row + i) for i in range(n)]
        assert [d for d, _ in covered] == list(range(h))
        assert [p for _, p in covered] == list(range(pos0 - h, pos0))
    assert ends == seq_len


@pytest.mark.parametrize("seq_len,world,window", CASES)
def test_sends_mirror_receives(seq_len, world, window):
    sent = sorted((r, dst, src_row, dst_row, n) for r in range(world)
                  for dst, src_row, dst_row, n in cp.halo_destinations(seq_len, world, r, window))
    recv = sorted((src, r, src_row, dst_row, n) for r in range(world)
                  for src, src_row, dst_row, n in cp.halo_sources(seq_len, world, r, window))
    assert sent == recv


def test_window_one_needs_no_halo():
    for r in range(4):
        assert cp.halo_sources(100, 4, r, 1) == []


def _full_kv(seq_len):
    g = torch.Generator().manual_seed(77)
    k = torch.randn((seq_len, 2, 192), generator=g).to(torch.bfloat16)
    v = torch.randn((seq_len, 2, 128), generator=g).to(torch.bfloat16)
    return k, v


def _rank(rank, world, port, seq_len, window, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        k, v = _full_kv(seq_len)
        pos0, length = cp.shard_bounds(seq_len, world, rank)
        h = cp.halo_len(pos0, window)
        kb = torch.full((h + length, 2, 192), float("nan"), dtype=torch.bfloat16)
        vb = torch.full((h + length, 2, 128), float("nan"), dtype=torch.bfloat16)
        kb[h:] = k[pos0:pos0 + length]
        vb[h:] = v[pos0:pos0 + length]
        got = cp.exchange_halo(kb, vb, seq_len, window)
        out[rank] = (got == h and torch.equal(kb, k[pos0 - h:pos0 + length])
                     and torch.equal(vb, v[pos0 - h:pos0 + length]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("seq_len,world,window", [(1000, 2, 128), (300, 3, 128), (90, 3, 0)])
def test_gloo_exchange_fills_every_halo(seq_len, world, window):
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank, args=(world, port, seq_len, window, out), nprocs=world,
                           start_method="spawn", join=True)
        res = dict(out)
    assert res == {r: True for r in range(world)}


def test_single_process_assembly_matches_the_sequence():
    seq_len, world, window = 300, 4, 128
    k, _ = _full_kv(seq_len)
    own = [k[p:p + n] for p, n in (cp.shard_bounds(seq_len, world, r) for r in range(world))]
    for r in range(world):
        pos0, length = cp.shard_bounds(seq_len, world, r)
        h = cp.halo_len(pos0, window)
        assert torch.equal(cp.halo_from_shards(own, seq_len, window, r), k[pos0 - h:pos0 + length])
