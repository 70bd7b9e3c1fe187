"""hattn_decode_static_scratch(): the decode / verify step for callers that
cannot allocate device memory (a host framework that owns every device
allocation through its own pool, or a serving loop whose memory budget is
fixed at start-up), so they cannot hand hattn_decode() a workspace.

It is checked through the C ABI against hattn_decode() with a caller
workspace, on two calls in a row (the shared scratch array keeps the first
call's contents when the second starts).  This file is collected last so that
a run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import global_attention_sinks_gqa_b300 as ha
import synth
from gpu_util import TOL_LSE, TOL_MAXABS, TOL_RELL2, fill_cache

pytestmark = pytest.mark.gpu


def _run_both(d, cap, is_ring, seed):
    dev = torch.device("cuda")
    B, T, hq, hkv = d.B, d.T, d.hq, d.hkv
    kc, vc = fill_cache(d, cap, is_ring)
    q, sink = d.q.to(dev), d.sink.to(dev)
    sl = torch.tensor(d.seqlens, dtype=torch.int32, device=dev)
    maxk = max(d.seqlens)
    need = ha.hattn_decode_workspace_size(B, T, hq, hkv, 128, maxk, d.window, cap, int(is_ring))
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    ref_o = torch.empty((B, T, hq, 128), dtype=torch.bfloat16, device=dev)
    ref_l = torch.empty((B, T, hq), dtype=torch.float32, device=dev)
    st = ha.hattn_decode(q, kc, vc, sl, sink, ref_o, ref_l, B, T, hq, hkv, 192, 128, cap,
                         int(is_ring), d.window, maxk, 64, d.rope_base, d.scale, ws, ws.numel())
    assert st == ha.HATTN_OK
    results = []
    for _ in range(2):  # two calls in a row share the one scratch array
        o = torch.full((B, T, hq, 128), float("nan"), dtype=torch.bfloat16, device=dev)
        l = torch.full((B, T, hq), float("nan"), dtype=torch.float32, device=dev)
        st = ha.hattn_decode_static_scratch(q, kc, vc, sl, sink, o, l, B, T, hq, hkv, 192, 128,
                                            cap, int(is_ring), d.window, maxk, 64, d.rope_base,
                                            d.scale)
        assert st == ha.HATTN_OK, ha.status_string(st)
        results.append((o, l))
    torch.cuda.synchronize()
    assert ha.hattn_check_device_status() == ha.HATTN_OK
    for o, l in results:
        a = o.float().cpu().double().numpy()
        b = ref_o.float().cpu().double().numpy()
        assert np.isfinite(a).all() and np.isfinite(l.cpu().numpy()).all()
        assert np.abs(a - b).max() <= TOL_MAXABS
        assert np.linalg.norm(a - b) / np.linalg.norm(b) <= TOL_RELL2
        assert (l - ref_l).abs().max().item() <= TOL_LSE
    return need


def test_static_scratch_decode_matches_workspace_decode():
    # global layer split over several 2048-key chunks: the scratch is used
    d = synth.decode_case([5000, 700, 4100, 2049], 4, 64, 4, window=0, rope_base=5e6, seed=1200)
    need = _run_both(d, 5004, False, 1200)
    assert 0 < need <= 32 * 1024 * 1024
    # a window layer over a ring fits one chunk: no scratch needed
    d = synth.decode_case([300, 131, 9], 3, 64, 8, window=128, rope_base=1e4, seed=1201)
    assert _run_both(d, 130, True, 1201) == 0


def test_static_scratch_rejects_steps_beyond_its_size():
    dev = torch.device("cuda")
    B, T, hq, hkv, maxk = 64, 4, 64, 4, 65536  # 1M partial rows: far beyond 32 MiB
    assert ha.hattn_decode_workspace_size(B, T, hq, hkv, 128, maxk, 0, maxk, 0) > 32 * 1024 * 1024
    fake = torch.empty(16, dtype=torch.uint8, device=dev)
    st = ha.hattn_decode_static_scratch(fake, fake, fake, fake, fake, fake, fake, B, T, hq, hkv,
                                        192, 128, maxk, 0, 0, maxk, 64, 5e6, 0.07)
    assert st == ha.HATTN_ERR_WORKSPACE
