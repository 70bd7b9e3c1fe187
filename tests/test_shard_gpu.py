"""Context-parallel shards of one sequence against the oracle on the whole
sequence (one GPU).

Each shard runs hattn_prefill_shard over its queries and its halo + own keys,
at absolute RoPE positions; the halo buffers are assembled in this process
with the same bookkeeping the exchange uses (halo_from_shards), standing in
for the point-to-point step that needs several GPUs.  The shards' rows must
match the oracle's rows of the unsharded sequence.
"""
import numpy as np
import pytest
import torch

import global_attention_sinks_gqa_b300 as ha
from global_attention_sinks_gqa_b300 import context_parallel as cp
import synth
from gpu_util import compare, oracle_prefill

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seq_len,world,G,window,base", [
    (1000, 2, 8, 128, 1e4),    # the window layer's group size, shards longer than the halo
    (700, 3, 16, 128, 1e4),    # G = 16 (one-block window units)
    (300, 4, 8, 128, 1e4),     # shards of 75 tokens: halos span two earlier shards
    (900, 3, 4, 64, 1e4),      # G = 4, two-block window units
    (600, 3, 16, 0, 5e6),      # a global layer: the whole history is the halo
    (257, 5, 2, 1, 1e4),       # window 1: no halo at all
])
def test_shards_match_the_unsharded_sequence(seq_len, world, G, window, base):
    dev = torch.device("cuda")
    c = synth.prefill_case([seq_len], 2 * G, 2, window=window, rope_base=base,
                           seed=1100 + seq_len + world)
    q, k, v, sink = c.q.to(dev), c.k.to(dev), c.v.to(dev), c.sink.to(dev)
    bounds = [cp.shard_bounds(seq_len, world, r) for r in range(world)]
    own_k = [k[p:p + n] for p, n in bounds]
    own_v = [v[p:p + n] for p, n in bounds]
    outs, lses = [], []
    for r, (pos0, length) in enumerate(bounds):
        h = cp.halo_len(pos0, window)
        kb = cp.halo_from_shards(own_k, seq_len, window, r)
        vb = cp.halo_from_shards(own_v, seq_len, window, r)
        o, l = ha.prefill_shard(q[pos0:pos0 + length].contiguous(), kb, vb, sink, pos0=pos0,
                                halo=h, window=window, rope_base=base, softmax_scale=c.scale)
        outs.append(o)
        lses.append(l)
    torch.cuda.synchronize()
    ha.check_device_status()
    o_ref, l_ref = oracle_prefill(c)
    compare(torch.cat(outs), torch.cat(lses), o_ref, l_ref,
            f"{world} shards of {seq_len}, G={G}, W={window}")


def test_shard_with_a_longer_halo_than_needed():
    """A halo longer than window - 1 (keys the window cannot reach) changes
    nothing: the extra keys are masked."""
    dev = torch.device("cuda")
    seq_len, pos0, G, window = 800, 400, 8, 128
    c = synth.prefill_case([seq_len], 2 * G, 2, window=window, rope_base=1e4, seed=1190)
    q, k, v, sink = c.q.to(dev), c.k.to(dev), c.v.to(dev), c.sink.to(dev)
    res = []
    for h in (127, 300):
        o, l = ha.prefill_shard(q[pos0:].contiguous(), k[pos0 - h:].contiguous(),
                                v[pos0 - h:].contiguous(), sink, pos0=pos0, halo=h,
                                window=window, rope_base=1e4, softmax_scale=c.scale)
        res.append((o, l))
    torch.cuda.synchronize()
    o_ref, l_ref = oracle_prefill(c, rows=np.arange(pos0, seq_len))
    for o, l in res:
        compare(o, l, o_ref, l_ref, "longer halo")
