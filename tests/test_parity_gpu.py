"""CUDA path vs the fp64 oracle, element by element, on the same seeded inputs.

Small cases are compared in full; the full-size workloads are compared on
sampled rows (rows are independent, so a sampled row is exact).
"""
import math

import numpy as np
import pytest
import torch

import global_attention_sinks_gqa_b300 as ha
import oracle
import synth
from gpu_util import compare, fill_cache, gpu_prefill, oracle_prefill

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ prefill
def test_prefill_tiny_swa_config():
    """batch 1, seq 512, 8 query heads / 1 KV head, W = 128, base 1e4, seed 0."""
    cfg = synth.CONFIGS["tiny_swa"]
    c = synth.prefill_case(cfg["seqlens"], cfg["hq"], cfg["hkv"], window=cfg["window"],
                           rope_base=cfg["rope_base"], seed=cfg["seed"])
    out, lse = gpu_prefill(c)
    o_ref, l_ref = oracle_prefill(c)
    compare(out, lse, o_ref, l_ref, "tiny swa")


RAGGED = [1, 127, 128, 129, 255, 1000, 3, 16, 17]


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("window,base", [(128, 1e4), (0, 5e6)])
def test_prefill_ragged_varlen(G, window, base):
    c = synth.prefill_case(RAGGED, 2 * G, 2, window=window, rope_base=base, seed=100 + G)
    out, lse = gpu_prefill(c)
    o_ref, l_ref = oracle_prefill(c)
    compare(out, lse, o_ref, l_ref, f"ragged G={G} W={window}")


@pytest.mark.parametrize("window", [1, 2, 7, 16, 100, 200, 255, 256, 257, 300, 1000])
def test_prefill_window_widths(window):
    c = synth.prefill_case([700, 301], 16, 2, window=window, rope_base=1e4, seed=200 + window)
    out, lse = gpu_prefill(c)
    o_ref, l_ref = oracle_prefill(c)
    compare(out, lse, o_ref, l_ref, f"W={window}")


@pytest.mark.parametrize("G,window", [(4, 5), (4, 64), (4, 97), (2, 1), (2, 16), (2, 33),
                                      (16, 130), (16, 145)])
def test_prefill_window_two_block_tiles(G, window):
    """Window units whose band (W - 1 + 256 / G keys) fits two 80-key blocks
    but not the one-block tile: G = 4 up to W = 97, G = 2 up to W = 33, and
    G = 16 just past the 144-key one-block band (W = 130 .. 145); ragged
    lengths so that tiles end mid-block."""
    c = synth.prefill_case(RAGGED, 2 * G, 2, window=window, rope_base=1e4, seed=800 + G + window)
    out, lse = gpu_prefill(c)
    o_ref, l_ref = oracle_prefill(c)
    compare(out, lse, o_ref, l_ref, f"two-block window tiles G={G} W={window}")


def test_prefill_window_covering_sequence_is_global():
    c = synth.prefill_case([600], 8, 1, window=600, rope_base=1e4, seed=300)
    out_w, lse_w = gpu_prefill(c)
    c.window = 0
    out_g, lse_g = gpu_prefill(c)
    assert torch.equal(out_w, out_g) and torch.equal(lse_w, lse_g)
    o_ref, l_ref = oracle_prefill(c)
    compare(out_w, lse_w, o_ref, l_ref, "W=S")


@pytest.mark.parametrize("window,base,sink_mean,sink_std", [
    (128, 1e4, 6.0, 2.0),    # SWA: sink weight comparable to the window's mass
    (0, 5e6, 8.0, 2.0),      # GA: sinks near the row log-sum-exp (~7-8 at S ~ 1500)
    (0, 5e6, 12.0, 0.5),     # sink dominates
    (64, 1e4, -30.0, 1.0),   # sink negligible
])
def test_prefill_sink_stress(window, base, sink_mean, sink_std):
    c = synth.prefill_case([1500, 77], 16, 1, window=window, rope_base=base, seed=400,
                           sink_mean=sink_mean, sink_std=sink_std)
    out, lse = gpu_prefill(c)
    o_ref, l_ref = oracle_prefill(c)
    compare(out, lse, o_ref, l_ref, f"sink N({sink_mean},{sink_std})")
    # the sink is visible: dropping it would move the output by far more than the tolerance
    o0, _ = oracle.prefill(c.q, c.k, c.v, torch.full((16,), -math.inf),
                           c.cu_seqlens.tolist(), window=window, rope_base=base, scale=c.scale)
    if sink_mean > 0:
        assert np.abs(o0 - o_ref).max() > 0.1


@pytest.mark.parametrize("G", [8, 16])
def test_prefill_many_short_sequences(G):
    """More sequences than the kernel caches offsets for, most shorter than
    one unit of the sliding-window path."""
    rs = np.random.RandomState(600 + G)
    lens = [int(x) for x in rs.randint(1, 90, size=150)] + [700]
    c = synth.prefill_case(lens, 2 * G, 2, window=128, rope_base=1e4, seed=600 + G)
    out, lse = gpu_prefill(c)
    o_ref, l_ref = oracle_prefill(c)
    compare(out, lse, o_ref, l_ref, f"150 short sequences G={G}")


@pytest.mark.parametrize("hkv,window,lens", [(96, 0, [130, 57]), (96, 128, [200]),
                                              (520, 128, [70, 41])])
def test_prefill_many_kv_heads(hkv, window, lens):
    """G = 1 with many KV heads: the key-rotation pass packs whole tokens
    into a block (96 heads: 5 tokens of 384 tasks; 520 heads: one token whose
    2080 tasks take the block two rounds)."""
    c = synth.prefill_case(lens, hkv, hkv, window=window, rope_base=1e4, seed=610 + hkv)
    out, lse = gpu_prefill(c)
    o_ref, l_ref = oracle_prefill(c)
    compare(out, lse, o_ref, l_ref, f"hkv {hkv} window {window}")


@pytest.mark.parametrize("G,window", [(4, 64), (16, 0), (8, 128), (16, 128)])
def test_prefill_many_units_per_cta(G, window):
    """60 short sequences and 16 KV heads: every CTA runs a string of units
    of one or two key blocks back to back (W = 64 at G = 4: 80-key blocks;
    the global layer at G = 16), so the K_0 barriers of the K stages turn
    over at every unit; at W = 128 (one-block units) full and ragged tiles
    alternate, so O leaves by TMA stores and by direct stores in turn."""
    rs = np.random.RandomState(1800 + G)
    lens = [int(x) for x in rs.randint(1, 200, size=60)]
    c = synth.prefill_case(lens, G * 16, 16, window=window, rope_base=1e4 if window else 5e6,
                           seed=1800 + G)
    out, lse = gpu_prefill(c)
    o_ref, l_ref = oracle_prefill(c)
    compare(out, lse, o_ref, l_ref, f"many units per CTA G={G} W={window}")


@pytest.mark.parametrize("G", [8, 16])
def test_prefill_output_at_16_byte_offset(G):
    """out 16- but not 32-byte aligned, inside a NaN-filled buffer: the O
    quarters stored by TMA and those stored directly (16-byte stores then)
    land in place, and nothing outside out is written."""
    c = synth.prefill_case([700, 333], 8 * G, 8, window=128, rope_base=1e4, seed=670 + G)
    dev = torch.device("cuda")
    n = c.q.shape[0] * c.q.shape[1] * 128
    buf = torch.full((n + 8 + 64,), float("nan"), dtype=torch.bfloat16, device=dev)
    out = buf[8:8 + n].view(c.q.shape[0], c.q.shape[1], 128)
    assert out.data_ptr() % 32 == 16
    lse = torch.empty(c.q.shape[0], c.q.shape[1], dtype=torch.float32, device=dev)
    ha.prefill(c.q.to(dev), c.k.to(dev), c.v.to(dev), c.sink.to(dev), c.cu_seqlens.to(dev),
               max_seqlen=c.max_seqlen, window=c.window, rope_base=c.rope_base,
               softmax_scale=c.scale, out=out, lse=lse)
    torch.cuda.synchronize()
    ha.check_device_status()
    assert torch.isnan(buf[:8]).all() and torch.isnan(buf[8 + n:]).all()
    o_ref, l_ref = oracle_prefill(c)
    compare(out, lse, o_ref, l_ref, f"out at a 16-byte offset G={G}")


@pytest.mark.parametrize("G,window", [(8, 128), (16, 128), (8, 64)])
def test_prefill_window_max_jumps_late_in_band(G, window):
    """Each key is 0.8 x the query of its token's first head in the group, so
    that head's rows have their largest logit (~11, against ~2 elsewhere) on
    the diagonal, past the first half of a one-block band: the softmax moves
    its max after half 1 has been taken and scales half 1's weights down by
    far more than 2^8."""
    lens = [700, 333]
    c = synth.prefill_case(lens, 2 * G, 2, window=window, rope_base=1e4, seed=650 + G + window)
    c.k = (0.8 * c.q.float()[:, ::G, :]).to(torch.bfloat16).contiguous()
    out, lse = gpu_prefill(c)
    o_ref, l_ref = oracle_prefill(c)
    compare(out, lse, o_ref, l_ref, f"growing keys G={G} W={window}")


def test_prefill_repeatable_and_independent_of_lse_pointer():
    c = synth.prefill_case([1000, 500], 64, 8, window=128, rope_base=1e4, seed=500)
    out1, lse1 = gpu_prefill(c)
    out2, lse2 = gpu_prefill(c)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    dev = torch.device("cuda")
    out3, lse3 = ha.prefill(c.q.to(dev), c.k.to(dev), c.v.to(dev), c.sink.to(dev),
                            c.cu_seqlens.to(dev), max_seqlen=1000, window=128, rope_base=1e4,
                            softmax_scale=c.scale, with_lse=False)
    torch.cuda.synchronize()
    assert lse3 is None and torch.equal(out3, out1)


def _sample_rows(S, n_mid, seed):
    rs = np.random.RandomState(seed)
    mid = rs.choice(np.arange(64, S - 64), size=n_mid, replace=False)
    return np.unique(np.concatenate([np.arange(64), mid, np.arange(S - 64, S)]))


@pytest.mark.parametrize("name,n_mid", [("swa_prefill_32k", 512), ("ga_prefill_32k", 96)])
def test_prefill_full_size_sampled(name, n_mid):
    """The bench workloads at full size (seq 32768, 64 query heads), sampled rows."""
    cfg = synth.CONFIGS[name]
    dev = torch.device("cuda")
    c = synth.prefill_case(cfg["seqlens"], cfg["hq"], cfg["hkv"], window=cfg["window"],
                           rope_base=cfg["rope_base"], seed=cfg["seed"], device=dev)
    out, lse = ha.prefill(c.q, c.k, c.v, c.sink, c.cu_seqlens, max_seqlen=c.max_seqlen,
                          window=c.window, rope_base=c.rope_base, softmax_scale=c.scale)
    torch.cuda.synchronize()
    ha.check_device_status()
    S = c.total
    rows = _sample_rows(S, n_mid, cfg["seed"])
    if cfg["window"] == 0:  # a global row needs every earlier key: keep the oracle's work small
        rows = np.unique(np.concatenate([np.arange(8), rows[rows >= S - 8],
                                         _sample_rows(S, n_mid, 9)[64:64 + n_mid]]))
    cpu = synth.PrefillCase(c.q.cpu(), c.k.cpu(), c.v.cpu(), c.sink.cpu(), c.cu_seqlens.cpu(),
                            c.seqlens, c.hq, c.hkv, c.window, c.rope_base, c.scale)
    o_ref, l_ref = oracle_prefill(cpu, rows=rows)
    idx = torch.tensor(rows, device=dev)
    compare(out[idx], lse[idx], o_ref, l_ref, name)


# ------------------------------------------------------------------ append / decode
def test_append_writes_rotated_keys_into_slots():
    B, T, hkv, cap = 3, 4, 2, 131
    g = torch.Generator().manual_seed(600)
    k_new = torch.randn((B, T, hkv, 192), generator=g).to(torch.bfloat16)
    v_new = torch.randn((B, T, hkv, 128), generator=g).to(torch.bfloat16)
    start = [0, 129, 5000]  # ring wrap-around at 131 for the second and third
    dev = torch.device("cuda")
    for is_ring, base in [(True, 1e4), (False, 5e6)]:
        capx = cap if is_ring else 6000
        kc = torch.full((B, hkv, capx, 192), 7.0, dtype=torch.bfloat16, device=dev)
        vc = torch.full((B, hkv, capx, 128), 7.0, dtype=torch.bfloat16, device=dev)
        sp = torch.tensor(start, dtype=torch.int32, device=dev)
        ha.rope_kv_append(k_new.to(dev), v_new.to(dev), sp, kc, vc, is_ring=is_ring,
                          rope_base=base)
        torch.cuda.synchronize()
        ha.check_device_status()
        kc_h, vc_h = kc.cpu(), vc.cpu()
        written = torch.zeros((B, capx), dtype=torch.bool)
        for b in range(B):
            for t in range(T):
                pos = start[b] + t
                slot = pos % cap if is_ring else pos
                written[b, slot] = True
                for h in range(hkv):
                    ref = oracle.rope(k_new[b, t, h][None], [pos], rope_base=base)[0]
                    row = kc_h[b, h, slot]
                    rot = row[:64].view(torch.int16).view(torch.float16).double().numpy()
                    # fp16 keeps 11 significant bits: half-ulp rounding + fp32 work
                    assert np.all(np.abs(rot - ref[:64]) <= np.abs(ref[:64]) * 2.0 ** -11 + 1e-6)
                    assert torch.equal(row[64:], k_new[b, t, h, 64:])
                    assert torch.equal(vc_h[b, h, slot], v_new[b, t, h])
        untouched = ~written
        assert (kc_h.permute(0, 2, 1, 3)[untouched] == 7.0).all()
        assert (vc_h.permute(0, 2, 1, 3)[untouched] == 7.0).all()


def _decode_compare(d, cap, is_ring, what, init=0.0):
    dev = torch.device("cuda")
    kc, vc = fill_cache(d, cap, is_ring, init=init)
    sl = torch.tensor(d.seqlens, dtype=torch.int32, device=dev)
    out, lse = ha.decode(d.q.to(dev), kc, vc, sl, d.sink.to(dev), max_seqlen_k=max(d.seqlens),
                         window=d.window, is_ring=is_ring, rope_base=d.rope_base,
                         softmax_scale=d.scale)
    torch.cuda.synchronize()
    ha.check_device_status()
    o_ref, l_ref = oracle.decode(d.q, d.k_hist, d.v_hist, d.seqlens, d.sink, window=d.window,
                                 rope_base=d.rope_base, scale=d.scale)
    return compare(out, lse, o_ref, l_ref, what)


@pytest.mark.parametrize("T", [1, 2, 3, 4, 6, 8])
@pytest.mark.parametrize("G", [1, 8, 16])
def test_decode_swa_ring(T, G):
    lens = [T, T + 1, 100, 130, 131, 132, 500, 1000]
    d = synth.decode_case(lens, T, G * 2, 2, window=128, rope_base=1e4, seed=700 + T + G)
    _decode_compare(d, 128 + T - 1, True, f"swa ring T={T} G={G}")


@pytest.mark.parametrize("T", [1, 4, 8])
@pytest.mark.parametrize("G", [4, 16])
def test_decode_ga_linear_multi_chunk(T, G):
    lens = [T, 64, 1023, 1024, 1025, 2048, 2049, 5000]  # 1 to 3 chunks of 2048
    d = synth.decode_case(lens, T, G * 2, 2, window=0, rope_base=5e6, seed=800 + T + G)
    _decode_compare(d, max(lens) + 3, False, f"ga T={T} G={G}")


def test_decode_many_short_items():
    """150 sequences of one to three 64-slot blocks, 16 KV heads: every CTA of
    the split-KV kernel takes a run of short items back to back, so its K / V
    stages and its per-item epilogue barrier turn over at every item."""
    rs = np.random.RandomState(1700)
    lens = [int(x) for x in rs.randint(2, 190, size=150)]
    d = synth.decode_case(lens, 2, 4 * 16, 16, window=0, rope_base=5e6, seed=1700)
    _decode_compare(d, 192, False, "many short items")


@pytest.mark.parametrize("cap,window,T,lens", [
    (300, 128, 4, [4, 131, 299, 300, 301, 1000, 1234]),    # ring larger than W + T - 1
    (2100, 2000, 2, [2, 2100, 2101, 5000, 777]),            # ring over two chunks of 2048
    (5003, 5000, 4, [5003, 9000, 4, 12345]),                # ring over three chunks
])
def test_decode_ring_capacities(cap, window, T, lens):
    d = synth.decode_case(lens, T, 32, 2, window=window, rope_base=1e4, seed=1000 + cap)
    _decode_compare(d, cap, True, f"ring cap={cap} W={window} T={T}")


@pytest.mark.parametrize("window,T", [(128, 4), (1000, 3), (3000, 4)])
def test_decode_window_over_linear_cache(window, T):
    lens = [T, 129, 1002, 1500, 3003, 6000]
    d = synth.decode_case(lens, T, 32, 2, window=window, rope_base=1e4, seed=1100 + window)
    _decode_compare(d, max(lens) + 5, False, f"linear cache W={window} T={T}")


@pytest.mark.parametrize("cap,window,T,lens", [
    (131, 128, 4, [5, 60, 130, 400]),          # ring: slots past L never written
    (300, 128, 2, [2, 299, 700]),              # general ring path
    (6000, 0, 4, [3000, 100, 5999, 4]),        # linear cache: the tail past L
])
def test_decode_unwritten_slots_hold_nan(cap, window, T, lens):
    """Cache slots nobody wrote may hold anything, NaN included: a key there
    has weight 0 and must not turn the output into 0 * NaN."""
    is_ring = window > 0
    d = synth.decode_case(lens, T, 32, 2, window=window, rope_base=1e4 if is_ring else 5e6,
                          seed=1300 + cap)
    _decode_compare(d, cap, is_ring, f"NaN-filled cache cap={cap}", init=float("nan"))


def _append_step(d, cap, is_ring, init=0.0):
    """Caches holding each sequence's history before its T new tokens, and
    those tokens' un-rotated K / V as [B, T, hkv, d]."""
    dev = torch.device("cuda")
    T = d.q.shape[1]
    upto = [L - T for L in d.seqlens]
    kc, vc = fill_cache(d, cap, is_ring, upto=upto, init=init)
    k_new = torch.stack([d.k_hist[b, L - T:L] for b, L in enumerate(d.seqlens)]).to(dev)
    v_new = torch.stack([d.v_hist[b, L - T:L] for b, L in enumerate(d.seqlens)]).to(dev)
    sl = torch.tensor(d.seqlens, dtype=torch.int32, device=dev)
    return kc, vc, k_new.contiguous(), v_new.contiguous(), sl


@pytest.mark.parametrize("cap,window,T,G,lens", [
    (131, 128, 4, 8, [4, 5, 100, 130, 131, 132, 500, 1000]),   # append inside the ring kernel
    (128, 128, 1, 8, [1, 2, 127, 128, 129, 700]),
    (130, 128, 3, 4, [3, 64, 129, 130, 131, 4000]),
    (16, 16, 1, 2, [1, 15, 16, 17, 33]),
    (135, 128, 8, 4, [8, 9, 134, 135, 136, 900]),              # 8 tokens, 32 rows: ring kernel
    (135, 128, 8, 16, [8, 9, 134, 135, 136, 900]),             # 128 rows: the general kernel
    (300, 128, 4, 8, [4, 131, 299, 300, 301, 1234]),           # append kernel, then the step
    (0, 0, 4, 16, [4, 100, 2048, 2049, 5000]),                  # linear cache
])
def test_decode_append_is_append_then_decode(cap, window, T, G, lens):
    """hattn_decode_append == hattn_rope_kv_append at seqlens - T followed by
    hattn_decode: the same cache bytes and the same outputs, bit for bit; and
    the outputs match the oracle."""
    is_ring = window > 0
    cap = cap or max(lens) + 3
    base = 1e4 if is_ring else 5e6
    d = synth.decode_case(lens, T, G * 2, 2, window=window, rope_base=base,
                          seed=1500 + cap + T)
    dev = torch.device("cuda")
    kc, vc, k_new, v_new, sl = _append_step(d, cap, is_ring)
    kc2, vc2 = kc.clone(), vc.clone()
    q, sink = d.q.to(dev), d.sink.to(dev)
    kw = dict(max_seqlen_k=max(lens), window=window, is_ring=is_ring, rope_base=base,
              softmax_scale=d.scale)
    out, lse = ha.decode_append(q, k_new, v_new, kc, vc, sl, sink, **kw)
    ha.rope_kv_append(k_new, v_new, sl - T, kc2, vc2, is_ring=is_ring, rope_base=base)
    out2, lse2 = ha.decode(q, kc2, vc2, sl, sink, **kw)
    torch.cuda.synchronize()
    ha.check_device_status()
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2), "cache bytes differ"
    assert torch.equal(out, out2) and torch.equal(lse, lse2), "outputs differ"
    o_ref, l_ref = oracle.decode(d.q, d.k_hist, d.v_hist, d.seqlens, d.sink, window=window,
                                 rope_base=base, scale=d.scale)
    compare(out, lse, o_ref, l_ref, f"decode_append cap={cap} T={T} G={G}")


def test_decode_steps_back_to_back_same_layer():
    """Three decode steps of one window layer issued back to back, no
    synchronisation between them: the window-ring kernel is launched as a
    programmatic dependent and may start while the step before it runs, yet
    every step must read the tokens the previous step appended to the ring."""
    dev = torch.device("cuda")
    T, G, hkv, cap, window, base, nsteps = 4, 8, 8, 131, 128, 1e4, 3
    rs = np.random.RandomState(1600)
    lens = [int(x) for x in rs.randint(3 * T, 900, size=32)] + [3 * T, 131 + 3 * T]
    d = synth.decode_case(lens, T, G * hkv, hkv, window=window, rope_base=base, seed=1601)
    kc, vc = fill_cache(d, cap, True, upto=[L - nsteps * T for L in lens])
    g = synth._gen(1602, "cpu")
    qs = [synth.randn_bf16((len(lens), T, G * hkv, synth.D_QK), g, "cpu") for _ in range(nsteps)]
    sink = d.sink.to(dev)
    outs = []
    for s in range(nsteps):  # step s appends positions L - (nsteps - s) T ..
        Ls = [L - (nsteps - 1 - s) * T for L in lens]
        k_new = torch.stack([d.k_hist[b, L - T:L] for b, L in enumerate(Ls)]).to(dev)
        v_new = torch.stack([d.v_hist[b, L - T:L] for b, L in enumerate(Ls)]).to(dev)
        outs.append((Ls, ha.decode_append(qs[s].to(dev), k_new.contiguous(), v_new.contiguous(),
                                          kc, vc, torch.tensor(Ls, dtype=torch.int32, device=dev),
                                          sink, max_seqlen_k=max(lens), window=window,
                                          is_ring=True, rope_base=base, softmax_scale=d.scale)))
    torch.cuda.synchronize()
    ha.check_device_status()
    for s, (Ls, (out, lse)) in enumerate(outs):
        o_ref, l_ref = oracle.decode(qs[s], d.k_hist, d.v_hist, Ls, d.sink, window=window,
                                     rope_base=base, scale=d.scale)
        compare(out, lse, o_ref, l_ref, f"back-to-back step {s}")


def test_decode_layers_back_to_back():
    """The decode step of three window layers and a global layer (separate
    caches) issued back to back, as a hybrid block runs them."""
    dev = torch.device("cuda")
    T = 4
    rs = np.random.RandomState(1610)
    lens = [int(x) for x in rs.randint(T, 3000, size=24)]
    layers = []
    for li, (window, hkv, base) in enumerate([(128, 8, 1e4)] * 3 + [(0, 4, 5e6)]):
        d = synth.decode_case(lens, T, 64, hkv, window=window, rope_base=base, seed=1611 + li)
        cap = 131 if window else max(lens) + 5
        kc, vc, k_new, v_new, sl = _append_step(d, cap, window > 0)
        layers.append((d, window, base, kc, vc, k_new, v_new, sl))
    res = []
    for d, window, base, kc, vc, k_new, v_new, sl in layers:
        res.append(ha.decode_append(d.q.to(dev), k_new, v_new, kc, vc, sl, d.sink.to(dev),
                                    max_seqlen_k=max(lens), window=window, is_ring=window > 0,
                                    rope_base=base, softmax_scale=d.scale))
    torch.cuda.synchronize()
    ha.check_device_status()
    for (d, window, base, *_), (out, lse) in zip(layers, res):
        o_ref, l_ref = oracle.decode(d.q, d.k_hist, d.v_hist, lens, d.sink, window=window,
                                     rope_base=base, scale=d.scale)
        compare(out, lse, o_ref, l_ref, f"layer chain W={window}")


def test_decode_append_unwritten_slots_hold_nan():
    """The fused append over a ring whose never-written slots hold NaN."""
    lens, T, cap = [4, 9, 60, 130, 131, 700], 4, 131
    d = synth.decode_case(lens, T, 16, 2, window=128, rope_base=1e4, seed=1600)
    dev = torch.device("cuda")
    kc, vc, k_new, v_new, sl = _append_step(d, cap, True, init=float("nan"))
    out, lse = ha.decode_append(d.q.to(dev), k_new, v_new, kc, vc, sl, d.sink.to(dev),
                                max_seqlen_k=max(lens), window=128, is_ring=True, rope_base=1e4,
                                softmax_scale=d.scale)
    torch.cuda.synchronize()
    ha.check_device_status()
    o_ref, l_ref = oracle.decode(d.q, d.k_hist, d.v_hist, d.seqlens, d.sink, window=128,
                                 rope_base=1e4, scale=d.scale)
    compare(out, lse, o_ref, l_ref, "decode_append NaN-filled ring")


@pytest.mark.parametrize("window,T", [(1, 1), (2, 2), (5, 4), (16, 1)])
def test_decode_tiny_rings(window, T):
    cap = window + T - 1
    d = synth.decode_case([T, T + 1, 7, 50], T, 64, 4, window=window, rope_base=1e4,
                          seed=1400 + window * 10 + T)
    _decode_compare(d, cap, True, f"tiny ring W={window} T={T}")


def test_decode_sink_stress():
    lens = [3000, 17, 4096]
    d = synth.decode_case(lens, 4, 64, 4, window=0, rope_base=5e6, seed=900, sink_mean=9.0,
                          sink_std=1.5)
    _decode_compare(d, 4100, False, "ga decode sink stress")
    d = synth.decode_case([400, 5], 4, 64, 8, window=128, rope_base=1e4, seed=901,
                          sink_mean=5.0, sink_std=1.0)
    _decode_compare(d, 131, True, "swa decode sink stress")


def test_decode_equals_prefill_last_rows():
    """The decode path on a cache equals the prefill path's last T rows."""
    L, T = 1500, 4
    for window, base, hkv, cap, ring in [(128, 1e4, 8, 131, True), (0, 5e6, 4, 2000, False)]:
        c = synth.prefill_case([L], 64, hkv, window=window, rope_base=base, seed=950)
        out_p, lse_p = gpu_prefill(c)
        d = synth.DecodeCase(c.q[L - T:][None], c.k[None], c.v[None], c.sink, [L], 64, hkv,
                             window, base, c.scale)
        dev = torch.device("cuda")
        kc, vc = fill_cache(d, cap, ring)
        out_d, lse_d = ha.decode(d.q.to(dev), kc, vc,
                                 torch.tensor([L], dtype=torch.int32, device=dev),
                                 c.sink.to(dev), max_seqlen_k=L, window=window, is_ring=ring,
                                 rope_base=base, softmax_scale=c.scale)
        torch.cuda.synchronize()
        diff = (out_d[0].float() - out_p[L - T:].float()).abs().max().item()
        assert diff <= 2e-2
        assert (lse_d[0] - lse_p[L - T:]).abs().max().item() <= 1e-3


def test_decode_full_size_config():
    """batch 64, 4 query tokens per sequence: SWA over a 131-slot ring (8 KV
    heads) and GA over lengths uniform in [8K, 64K] (4 KV heads).  The T new
    tokens go through the append kernel first, as in the bench step."""
    cfg = synth.CONFIGS["decode_b64_t4"]
    B, T = cfg["B"], cfg["T"]
    lens = synth.random_lengths(B, cfg["lens"][0], cfg["lens"][1], cfg["seed"])
    dev = torch.device("cuda")
    sample = sorted({int(np.argmax(lens)), int(np.argmin(lens)), 0, 17, 40})
    for layer, cap, ring in [("swa", 131, True), ("ga", 65536, False)]:
        p = cfg[layer]
        d = synth.decode_case(lens, T, p["hq"], p["hkv"], window=p["window"],
                              rope_base=p["rope_base"], seed=cfg["seed"], device=dev,
                              lmax=cfg["lens"][1])
        kc, vc = fill_cache(d, cap, ring, upto=[L - T for L in lens])
        idx = torch.arange(T, device=dev)
        k_new = torch.stack([d.k_hist[b, L - T + idx] for b, L in enumerate(lens)])
        v_new = torch.stack([d.v_hist[b, L - T + idx] for b, L in enumerate(lens)])
        sl = torch.tensor(lens, dtype=torch.int32, device=dev)
        ha.rope_kv_append(k_new, v_new, sl - T, kc, vc, is_ring=ring, rope_base=p["rope_base"])
        out, lse = ha.decode(d.q, kc, vc, sl, d.sink, max_seqlen_k=cfg["lens"][1],
                             window=p["window"], is_ring=ring, rope_base=p["rope_base"],
                             softmax_scale=d.scale)
        torch.cuda.synchronize()
        ha.check_device_status()
        for b in sample:
            L = lens[b]
            o_ref, l_ref = oracle.decode(d.q[b:b + 1].cpu(), d.k_hist[b:b + 1, :L].cpu(),
                                         d.v_hist[b:b + 1, :L].cpu(), [L], d.sink.cpu(),
                                         window=p["window"], rope_base=p["rope_base"],
                                         scale=d.scale)
            compare(out[b:b + 1], lse[b:b + 1], o_ref, l_ref, f"{layer} b={b} L={L}")
        del d, kc, vc
        torch.cuda.empty_cache()


def test_hybrid_block_256k_sampled():
    """One hybrid block at seq 262144: 5 SWA layers (64q/8kv, W=128, base 1e4)
    and 1 GA layer (64q/4kv, base 5e6), fresh inputs per layer, sampled rows."""
    cfg = synth.CONFIGS["hybrid_block_256k"]
    S = cfg["seqlens"][0]
    dev = torch.device("cuda")
    layers = [("swa", i) for i in range(cfg["n_swa"])] + [("ga", cfg["n_swa"])]
    for kind, li in layers:
        p = cfg[kind]
        c = synth.prefill_case([S], p["hq"], p["hkv"], window=p["window"],
                               rope_base=p["rope_base"], seed=cfg["seed"] * 100 + li, device=dev)
        out, lse = ha.prefill(c.q, c.k, c.v, c.sink, c.cu_seqlens, max_seqlen=S,
                              window=c.window, rope_base=c.rope_base, softmax_scale=c.scale)
        torch.cuda.synchronize()
        ha.check_device_status()
        if kind == "swa":
            rows = _sample_rows(S, 64, li)
        else:
            rows = np.array([0, 1, 130, 4097, 131071, S - 1])
        cpu = synth.PrefillCase(c.q.cpu(), c.k.cpu(), c.v.cpu(), c.sink.cpu(),
                                c.cu_seqlens.cpu(), c.seqlens, c.hq, c.hkv, c.window,
                                c.rope_base, c.scale)
        o_ref, l_ref = oracle_prefill(cpu, rows=rows)
        idx = torch.tensor(rows, device=dev)
        compare(out[idx], lse[idx], o_ref, l_ref, f"hybrid layer {li} ({kind})")
        del c, out, lse, cpu
        torch.cuda.empty_cache()


# ------------------------------------------------------------ prefill over a cached prefix
def _prefill_cached_case(prefixes, news, G, window, base, seed, init=0.0):
    """Sequences whose first prefixes[b] tokens sit in a linear cache and whose
    next news[b] tokens are new; returns the CUDA path's (out, lse) for the new
    tokens, the oracle's over each whole history, and the caches."""
    dev = torch.device("cuda")
    hq, hkv = 2 * G, 2
    Ls = [p + n for p, n in zip(prefixes, news)]
    d = synth.decode_case(Ls, 1, hq, hkv, window=window, rope_base=base, seed=seed)
    g = synth._gen(seed + 1, "cpu")
    q_new = [synth.randn_bf16((n, hq, synth.D_QK), g, "cpu") for n in news]
    B, cap = len(Ls), max(Ls) + 300
    kc = torch.full((B, hkv, cap, synth.D_QK), init, dtype=torch.bfloat16, device=dev)
    vc = torch.full((B, hkv, cap, synth.D_V), init, dtype=torch.bfloat16, device=dev)
    for b, P in enumerate(prefixes):
        if P:
            ha.rope_kv_append(d.k_hist[b:b + 1, :P].contiguous().to(dev),
                              d.v_hist[b:b + 1, :P].contiguous().to(dev),
                              torch.zeros(1, dtype=torch.int32, device=dev), kc[b:b + 1],
                              vc[b:b + 1], is_ring=False, rope_base=base)
    k_new = torch.cat([d.k_hist[b, P:P + n] for b, (P, n) in enumerate(zip(prefixes, news))])
    v_new = torch.cat([d.v_hist[b, P:P + n] for b, (P, n) in enumerate(zip(prefixes, news))])
    cu = torch.tensor([0] + list(np.cumsum(news)), dtype=torch.int32, device=dev)
    pre = torch.tensor(prefixes, dtype=torch.int32, device=dev)
    out, lse = ha.prefill_cached(torch.cat(q_new).to(dev), k_new.to(dev), v_new.to(dev), kc, vc,
                                 cu, pre, d.sink.to(dev), max_seqlen=max(news),
                                 max_prefix=max(prefixes), window=window, rope_base=base,
                                 softmax_scale=d.scale)
    torch.cuda.synchronize()
    ha.check_device_status()
    o_ref, l_ref = [], []
    for b, (P, n) in enumerate(zip(prefixes, news)):
        if n == 0:
            continue
        o, l = oracle.decode(q_new[b][None], d.k_hist[b:b + 1], d.v_hist[b:b + 1], [P + n],
                             d.sink, window=window, rope_base=base, scale=d.scale)
        o_ref.append(o[0])
        l_ref.append(l[0])
    return out, lse, np.concatenate(o_ref), np.concatenate(l_ref), (kc, vc, d, k_new, v_new)


@pytest.mark.parametrize("prefixes,news,G,window,base", [
    ([0, 100, 3000], [50, 300, 257], 16, 0, 5e6),       # global layer, ragged
    ([0, 1, 500], [700, 129, 64], 8, 128, 1e4),         # window over the cache (one block)
    ([2000, 0], [300, 1500], 4, 1000, 1e4),             # wide window (several blocks)
    ([4095, 17], [1, 2], 16, 0, 5e6),                   # one or two new tokens
])
def test_prefill_cached_prefix(prefixes, news, G, window, base):
    out, lse, o_ref, l_ref, _ = _prefill_cached_case(prefixes, news, G, window, base,
                                                     seed=1700 + G + window)
    compare(out, lse, o_ref, l_ref, f"cached prefix {prefixes} + {news} W={window}")


def test_prefill_cached_prefix_over_nan_slots():
    """Slots past the history hold NaN before the call: the appended keys and
    the zeroed value slots past them keep the output finite and exact."""
    out, lse, o_ref, l_ref, _ = _prefill_cached_case([37, 1200], [90, 333], 16, 0, 5e6,
                                                     seed=1800, init=float("nan"))
    compare(out, lse, o_ref, l_ref, "cached prefix over NaN slots")


def test_prefill_cached_appends_like_rope_kv_append():
    """The new tokens land in the caches exactly as hattn_rope_kv_append writes them."""
    prefixes, news = [10, 300], [40, 77]
    _, _, _, _, (kc, vc, d, k_new, v_new) = _prefill_cached_case(prefixes, news, 8, 128, 1e4,
                                                                 seed=1900)
    dev = torch.device("cuda")
    kc2, vc2 = torch.zeros_like(kc), torch.zeros_like(vc)
    off = 0
    for b, (P, n) in enumerate(zip(prefixes, news)):
        ha.rope_kv_append(k_new[off:off + n][None].to(dev), v_new[off:off + n][None].to(dev),
                          torch.tensor([P], dtype=torch.int32, device=dev), kc2[b:b + 1],
                          vc2[b:b + 1], is_ring=False, rope_base=1e4)
        assert torch.equal(kc[b, :, P:P + n], kc2[b, :, P:P + n])
        assert torch.equal(vc[b, :, P:P + n], vc2[b, :, P:P + n])
        assert (vc[b, :, P + n:P + n + 256] == 0).all()   # the zeroed tail
        off += n
    torch.cuda.synchronize()


def test_prefill_cached_without_prefix_matches_prefill():
    """Empty prefixes: the same attention as hattn_prefill of the new tokens."""
    news, G = [300, 129, 64], 8
    out, lse, o_ref, l_ref, (kc, vc, d, k_new, v_new) = _prefill_cached_case(
        [0, 0, 0], news, G, 128, 1e4, seed=2000)
    compare(out, lse, o_ref, l_ref, "cached prefix, none cached")


# ------------------------------------------------------------ paged caches
@pytest.mark.parametrize("page,G,window,base,T,lens", [
    (64, 16, 0, 5e6, 4, [4, 63, 64, 65, 700, 3000]),     # one or many pages, one chunk
    (128, 8, 128, 1e4, 4, [4, 200, 1000]),                # a window over pages
    (256, 16, 0, 5e6, 1, [5000, 9000, 130]),              # split-KV chunks over pages
])
def test_decode_append_paged(page, G, window, base, T, lens):
    """Paged caches (pages in shuffled order) hold the bytes of the contiguous
    caches, give their outputs (bit for bit without a window), and match the
    oracle."""
    dev = torch.device("cuda")
    d = synth.decode_case(lens, T, 2 * G, 2, window=window, rope_base=base,
                          seed=2100 + page + G + T)
    stride = (max(lens) + 3 + page - 1) // page
    kc, vc, k_new, v_new, sl = _append_step(d, stride * page, False)
    B, hkv = len(lens), 2
    num_pages = B * stride + 5
    rs = np.random.RandomState(2200 + page)
    table = torch.tensor(rs.permutation(num_pages)[:B * stride].reshape(B, stride),
                         dtype=torch.int32, device=dev)
    kp = torch.zeros((num_pages, hkv, page, synth.D_QK), dtype=torch.bfloat16, device=dev)
    vp = torch.zeros((num_pages, hkv, page, synth.D_V), dtype=torch.bfloat16, device=dev)
    for b in range(B):
        for lp in range(stride):
            kp[table[b, lp]] = kc[b, :, lp * page:(lp + 1) * page]
            vp[table[b, lp]] = vc[b, :, lp * page:(lp + 1) * page]
    q, sink = d.q.to(dev), d.sink.to(dev)
    kw = dict(max_seqlen_k=max(lens), window=window, rope_base=base, softmax_scale=d.scale)
    out_p, lse_p = ha.decode_append_paged(q, k_new, v_new, kp, vp, table, sl, sink, **kw)
    out_l, lse_l = ha.decode_append(q, k_new, v_new, kc, vc, sl, sink, is_ring=False, **kw)
    torch.cuda.synchronize()
    ha.check_device_status()
    if window == 0:  # same blocks as the contiguous cache: the same bits
        assert torch.equal(out_p, out_l) and torch.equal(lse_p, lse_l), "paged != contiguous"
    # (with a window the paged item starts on a 64-slot boundary, so its blocks
    # and hence its rounding differ from the contiguous cache's)
    for b in range(B):
        for lp in range(stride):
            assert torch.equal(kp[table[b, lp]], kc[b, :, lp * page:(lp + 1) * page])
            assert torch.equal(vp[table[b, lp]], vc[b, :, lp * page:(lp + 1) * page])
    o_ref, l_ref = oracle.decode(d.q, d.k_hist, d.v_hist, d.seqlens, d.sink, window=window,
                                 rope_base=base, scale=d.scale)
    compare(out_p, lse_p, o_ref, l_ref, f"paged decode page={page} G={G} W={window}")
