"""Failure detection without a GPU fault: a bounded device-side wait that runs
out ends the kernel normally and reports HATTN_ERR_TIMEOUT through the device
status word; device-resident arguments the host could not check are skipped
and reported.  The context stays usable afterwards."""
import pytest
import torch

import global_attention_sinks_gqa_b300 as ha
import synth
from gpu_util import compare, gpu_prefill, oracle_prefill

pytestmark = pytest.mark.gpu


def test_lost_arrival_times_out_and_context_survives():
    assert ha.hattn_check_device_status() == ha.HATTN_OK
    assert ha.hattn_set_wait_limit_ns(50_000_000) == ha.HATTN_OK  # 50 ms
    try:
        assert ha.hattn_selftest_lost_arrival() == ha.HATTN_OK
        assert ha.hattn_check_device_status() == ha.HATTN_ERR_TIMEOUT
        assert ha.hattn_check_device_status() == ha.HATTN_OK  # read clears it
    finally:
        ha.hattn_set_wait_limit_ns(0)
    c = synth.prefill_case([300], 8, 1, window=128, rope_base=1e4, seed=1000)
    out, lse = gpu_prefill(c)
    compare(out, lse, *oracle_prefill(c), "after timeout")


def test_device_side_length_check_skips_and_reports():
    dev = torch.device("cuda")
    B, T, hq, hkv, cap = 2, 2, 16, 1, 64
    q = torch.randn((B, T, hq, 192), device=dev).to(torch.bfloat16)
    kc = torch.zeros((B, hkv, cap, 192), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros((B, hkv, cap, 128), dtype=torch.bfloat16, device=dev)
    sink = torch.zeros(hq, device=dev)
    seqlens = torch.tensor([10, 200], dtype=torch.int32, device=dev)  # 200 > cap
    out = torch.full((B, T, hq, 128), 3.0, dtype=torch.bfloat16, device=dev)
    st = ha.hattn_decode(q, kc, vc, seqlens, sink, out, None, B, T, hq, hkv, 192, 128, cap, 0, 0,
                         cap, 64, 5e6, 0.07, None, 0)
    assert st == ha.HATTN_OK
    assert ha.hattn_check_device_status() == ha.HATTN_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (out[1] == 3.0).all()          # the bad sequence was not touched
    assert torch.isfinite(out[0].float()).all()


def test_append_position_beyond_linear_cache_is_reported():
    dev = torch.device("cuda")
    k = torch.randn((1, 2, 1, 192), device=dev).to(torch.bfloat16)
    v = torch.randn((1, 2, 1, 128), device=dev).to(torch.bfloat16)
    kc = torch.zeros((1, 1, 8, 192), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros((1, 1, 8, 128), dtype=torch.bfloat16, device=dev)
    pos = torch.tensor([7], dtype=torch.int32, device=dev)  # position 8 does not fit
    ha.rope_kv_append(k, v, pos, kc, vc, is_ring=False, rope_base=1e4)
    assert ha.hattn_check_device_status() == ha.HATTN_ERR_INVALID_ARG
    assert torch.equal(vc[0, 0, 7].cpu(), v[0, 0, 0].cpu())  # position 7 was written


def test_injected_launch_failure_leaves_outputs_untouched():
    """A launch failure injected on the host surfaces as HATTN_ERR_CUDA through
    the Python binding, writes nothing, and the next call runs normally."""
    dev = torch.device("cuda")
    c = synth.prefill_case([300], 16, 2, window=128, rope_base=1e4, seed=61, device=dev)
    kw = dict(max_seqlen=300, window=128, rope_base=1e4)
    ref, ref_lse = ha.prefill(c.q, c.k, c.v, c.sink, c.cu_seqlens, **kw)
    out = torch.full_like(ref, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    assert ha.hattn_test_fail_next_launches(1) == 0
    with pytest.raises(ha.HattnError) as e:
        ha.prefill(c.q, c.k, c.v, c.sink, c.cu_seqlens, out=out, lse=lse, **kw)
    assert e.value.status == ha.HATTN_ERR_CUDA
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all() and torch.isnan(lse).all()
    assert ha.hattn_test_fail_next_launches(0) == 0
    ha.prefill(c.q, c.k, c.v, c.sink, c.cu_seqlens, out=out, lse=lse, **kw)
    torch.cuda.synchronize()
    ha.check_device_status()
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
