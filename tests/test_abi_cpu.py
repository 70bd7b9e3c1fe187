"""The C-ABI library loads, exports every entry point include/hattn.h
declares, and rejects bad arguments on the host before touching the GPU."""
import ctypes
import os
import re

import pytest

import global_attention_sinks_gqa_b300 as ha
from global_attention_sinks_gqa_b300 import build as hbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    hbuild.build()
    return ha.load_library()


def header_functions():
    src = open(os.path.join(ROOT, "include", "hattn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hattn_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = header_functions()
    assert "hattn_prefill" in names and "hattn_decode" in names
    assert "hattn_rope_kv_append" in names
    for n in names:
        assert hasattr(lib, n), n
        assert n in ha.SIGNATURES, n


def test_version_and_status_strings(lib):
    assert ha.hattn_version() >= 100
    for code, name in [(0, "HATTN_OK"), (1, "HATTN_ERR_INVALID_ARG"),
                       (2, "HATTN_ERR_UNSUPPORTED"), (4, "HATTN_ERR_RING_TOO_SMALL"),
                       (5, "HATTN_ERR_TIMEOUT"), (6, "HATTN_ERR_WORKSPACE")]:
        assert ha.status_string(code) == name


def test_workspace_sizes(lib):
    # the keys' rotated dims 0..63 (fp16) rounded to 256 bytes, then 256 bytes
    # of work counter
    assert ha.hattn_prefill_workspace_size(32768, 8, 192) == 32768 * 8 * 64 * 2 + 256
    assert ha.hattn_prefill_workspace_size(3, 1, 192) == 512 + 256  # 384 rounded to 256
    # a ring window fits one chunk: no workspace
    assert ha.hattn_decode_workspace_size(64, 4, 64, 8, 128, 65536, 128, 131, 1) == 0
    # partial O and lse (each rounded to 256 bytes), then 256 bytes of work counter
    n = ha.hattn_decode_workspace_size(64, 4, 64, 4, 128, 65536, 0, 65536, 0)
    rows = 64 * 64 * 4 * 16  # 16 chunks of 4096 keys (caches beyond 16K keys)
    assert n == rows * 128 * 4 + rows * 4 + 256
    n = ha.hattn_decode_workspace_size(8, 4, 64, 4, 128, 10000, 0, 10000, 0)
    rows = 8 * 64 * 4 * 5  # 5 chunks of 2048 keys
    assert n == rows * 128 * 4 + rows * 4 + 256
    # a ring is cut by its capacity, not by the window
    assert ha.hattn_decode_workspace_size(2, 1, 16, 1, 128, 9000, 1000, 3000, 1) > 0
    assert ha.hattn_decode_workspace_size(2, 1, 16, 1, 128, 9000, 1000, 1000, 1) == 0


FAKE = 1 << 20  # a 16-byte aligned non-null "device pointer" never dereferenced


def _prefill(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, sink=FAKE, out=FAKE, lse=FAKE, batch=1,
                cu_seqlens=FAKE, total_tokens=512, max_seqlen=512, hq=8, hkv=1, dqk=192, dv=128,
                rope_dim=64, rope_base=1e4, window=128, softmax_scale=0.07, workspace=FAKE,
                workspace_bytes=512 * 192 * 2, stream=0)
    args.update(kw)
    return ha.hattn_prefill(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(hkv=3), ha.HATTN_ERR_INVALID_ARG),
    (dict(dqk=128), ha.HATTN_ERR_UNSUPPORTED),
    (dict(dv=64), ha.HATTN_ERR_UNSUPPORTED),
    (dict(rope_dim=32), ha.HATTN_ERR_UNSUPPORTED),
    (dict(hq=64, hkv=2), ha.HATTN_ERR_UNSUPPORTED),      # G = 32
    (dict(q=None), ha.HATTN_ERR_INVALID_ARG),
    (dict(q=FAKE + 8), ha.HATTN_ERR_INVALID_ARG),        # misaligned
    (dict(window=-1), ha.HATTN_ERR_INVALID_ARG),
    (dict(softmax_scale=0.0), ha.HATTN_ERR_INVALID_ARG),
    (dict(rope_base=float("nan")), ha.HATTN_ERR_INVALID_ARG),
    (dict(max_seqlen=513), ha.HATTN_ERR_INVALID_ARG),
    (dict(workspace_bytes=100), ha.HATTN_ERR_WORKSPACE),
    (dict(workspace=None), ha.HATTN_ERR_WORKSPACE),
    (dict(batch=0), ha.HATTN_ERR_INVALID_ARG),
])
def test_prefill_rejects_bad_arguments(lib, kw, code):
    assert _prefill(**kw) == code


def _decode(**kw):
    args = dict(q=FAKE, k_cache=FAKE, v_cache=FAKE, seqlens_k=FAKE, sink=FAKE, out=FAKE,
                lse=FAKE, B=64, T=4, hq=64, hkv=8, dqk=192, dv=128, cap=131, is_ring=1,
                window=128, max_seqlen_k=65536, rope_dim=64, rope_base=1e4, softmax_scale=0.07,
                workspace=None, workspace_bytes=0, stream=0)
    args.update(kw)
    return ha.hattn_decode(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(cap=130), ha.HATTN_ERR_RING_TOO_SMALL),          # needs W + T - 1 = 131
    (dict(cap=127, T=1), ha.HATTN_ERR_RING_TOO_SMALL),
    (dict(T=9, cap=136), ha.HATTN_ERR_UNSUPPORTED),          # up to 8 tokens per step
    (dict(T=0), ha.HATTN_ERR_INVALID_ARG),
    (dict(is_ring=1, window=0), ha.HATTN_ERR_INVALID_ARG),
    (dict(is_ring=0, window=0, hkv=4, cap=1000, max_seqlen_k=2000), ha.HATTN_ERR_INVALID_ARG),
    (dict(is_ring=0, window=0, hkv=4, cap=65536), ha.HATTN_ERR_WORKSPACE),
    (dict(hq=64, hkv=2), ha.HATTN_ERR_UNSUPPORTED),
    (dict(max_seqlen_k=3), ha.HATTN_ERR_INVALID_ARG),
    (dict(q=FAKE + 4), ha.HATTN_ERR_INVALID_ARG),
])
def test_decode_rejects_bad_arguments(lib, kw, code):
    assert _decode(**kw) == code


def test_decode_window_near_int_max_does_not_wrap(lib):
    """A window of INT_MAX ('no window') must not wrap window + T - 1 into a
    negative number: a ring would then pass the capacity check."""
    assert _decode(window=2**31 - 1) == ha.HATTN_ERR_RING_TOO_SMALL
    # over a linear cache such a window is global attention (same workspace need)
    assert _decode(is_ring=0, window=2**31 - 1, hkv=4, cap=65536) == ha.HATTN_ERR_WORKSPACE


@pytest.mark.parametrize("kw,code", [
    (dict(dqk=64), ha.HATTN_ERR_UNSUPPORTED),
    (dict(T=9), ha.HATTN_ERR_UNSUPPORTED),
    (dict(hq=64, hkv=5), ha.HATTN_ERR_INVALID_ARG),
    (dict(q=None), ha.HATTN_ERR_INVALID_ARG),
    (dict(), ha.HATTN_ERR_WORKSPACE),        # valid, but its partials exceed the array
])
def test_static_scratch_checks_arguments_before_its_size(lib, kw, code):
    """A malformed call to the allocation-free decode step reports its argument
    error even when its scratch need would also exceed the fixed array."""
    args = dict(q=FAKE, k_cache=FAKE, v_cache=FAKE, seqlens_k=FAKE, sink=FAKE, out=FAKE,
                lse=FAKE, B=64, T=4, hq=64, hkv=4, dqk=192, dv=128, cap=65536, is_ring=0,
                window=0, max_seqlen_k=65536, rope_dim=64, rope_base=5e6, softmax_scale=0.07,
                stream=0)
    args.update(kw)
    assert ha.hattn_decode_static_scratch(**args) == code


@pytest.mark.parametrize("kw,code", [
    (dict(T=0), ha.HATTN_ERR_INVALID_ARG),
    (dict(T=200, cap=131), ha.HATTN_ERR_INVALID_ARG),
    (dict(is_ring=2), ha.HATTN_ERR_INVALID_ARG),
    (dict(dqk=64), ha.HATTN_ERR_UNSUPPORTED),
    (dict(k_cache=None), ha.HATTN_ERR_INVALID_ARG),
])
def test_append_rejects_bad_arguments(lib, kw, code):
    args = dict(k_new=FAKE, v_new=FAKE, start_pos=FAKE, k_cache=FAKE, v_cache=FAKE, B=64, T=4,
                hkv=8, dqk=192, dv=128, cap=131, is_ring=1, rope_dim=64, rope_base=1e4, stream=0)
    args.update(kw)
    assert ha.hattn_rope_kv_append(**args) == code


def _prefill_cached(**kw):
    args = dict(q=FAKE, k_new=FAKE, v_new=FAKE, k_cache=FAKE, v_cache=FAKE, cu_seqlens=FAKE,
                prefix_lens=FAKE, sink=FAKE, out=FAKE, lse=FAKE, batch=2, total_tokens=512,
                max_seqlen=300, max_prefix=4096, cap=8192, hq=32, hkv=2, dqk=192, dv=128,
                rope_dim=64, rope_base=5e6, window=0, softmax_scale=0.07, workspace=FAKE,
                workspace_bytes=256, stream=0)
    args.update(kw)
    return ha.hattn_prefill_cached(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(workspace_bytes=128), ha.HATTN_ERR_WORKSPACE),    # the work counter needs 256 bytes
    (dict(workspace=None), ha.HATTN_ERR_WORKSPACE),
    (dict(prefix_lens=None), ha.HATTN_ERR_INVALID_ARG),
    (dict(k_cache=FAKE + 4), ha.HATTN_ERR_INVALID_ARG),      # misaligned
    (dict(max_prefix=-1), ha.HATTN_ERR_INVALID_ARG),
    (dict(cap=0), ha.HATTN_ERR_INVALID_ARG),
    (dict(max_seqlen=513), ha.HATTN_ERR_INVALID_ARG),
    (dict(dv=64), ha.HATTN_ERR_UNSUPPORTED),
])
def test_prefill_cached_rejects_bad_arguments(lib, kw, code):
    assert _prefill_cached(**kw) == code


def _decode_paged(**kw):
    args = dict(q=FAKE, k_new=FAKE, v_new=FAKE, k_pages=FAKE, v_pages=FAKE, block_table=FAKE,
                table_stride=256, num_pages=16384, page=256, seqlens_k=FAKE, sink=FAKE, out=FAKE,
                lse=FAKE, B=64, T=4, hq=64, hkv=4, dqk=192, dv=128, window=0,
                max_seqlen_k=65536, rope_dim=64, rope_base=5e6, softmax_scale=0.07,
                workspace=None, workspace_bytes=0, stream=0)
    args.update(kw)
    return ha.hattn_decode_append_paged(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(page=100), ha.HATTN_ERR_INVALID_ARG),              # pages hold whole 64-slot blocks
    (dict(page=0), ha.HATTN_ERR_INVALID_ARG),
    (dict(table_stride=0), ha.HATTN_ERR_INVALID_ARG),
    (dict(num_pages=0), ha.HATTN_ERR_INVALID_ARG),
    (dict(block_table=None), ha.HATTN_ERR_INVALID_ARG),
    (dict(block_table=FAKE + 2), ha.HATTN_ERR_INVALID_ARG),  # misaligned int32
    (dict(max_seqlen_k=65537), ha.HATTN_ERR_INVALID_ARG),     # past table_stride * page
    (dict(T=9), ha.HATTN_ERR_UNSUPPORTED),
    (dict(), ha.HATTN_ERR_WORKSPACE),                         # split chunks need a workspace
])
def test_decode_paged_rejects_bad_arguments(lib, kw, code):
    assert _decode_paged(**kw) == code


def _shard(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, sink=FAKE, out=FAKE, lse=FAKE, shard_tokens=1000,
                halo=127, pos0=4000, hq=64, hkv=8, dqk=192, dv=128, rope_dim=64, rope_base=1e4,
                window=128, softmax_scale=0.07, workspace=FAKE, workspace_bytes=1 << 30,
                stream=0)
    args.update(kw)
    return ha.hattn_prefill_shard(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(halo=126), ha.HATTN_ERR_INVALID_ARG),               # the window needs 127 rows
    (dict(halo=30, pos0=20), ha.HATTN_ERR_INVALID_ARG),       # more rows than positions
    (dict(halo=20, pos0=30), ha.HATTN_ERR_INVALID_ARG),       # needs min(127, 30) = 30
    (dict(window=0, halo=127), ha.HATTN_ERR_INVALID_ARG),     # global: the whole history
    (dict(pos0=2**31 - 500), ha.HATTN_ERR_INVALID_ARG),       # positions past INT_MAX
    (dict(shard_tokens=-1), ha.HATTN_ERR_INVALID_ARG),
    (dict(dqk=128), ha.HATTN_ERR_UNSUPPORTED),
    (dict(workspace_bytes=1000), ha.HATTN_ERR_WORKSPACE),
    (dict(k=FAKE + 8), ha.HATTN_ERR_INVALID_ARG),
    (dict(shard_tokens=0), ha.HATTN_OK),                      # nothing to do
])
def test_prefill_shard_rejects_bad_arguments(lib, kw, code):
    assert _shard(**kw) == code


def test_oracle_is_not_reachable_from_the_product():
    """The product package never imports the oracle."""
    pkg = os.path.join(ROOT, "global_attention_sinks_gqa_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in txt and "from oracle" not in txt, f
                assert "hattn_oracle" not in txt, f


def test_backward_workspace_size(lib):
    # rotated q and k dims 0..63 (bf16), delta (fp32), sink partials of
    # 32-token blocks (fp32), each rounded to 256 bytes
    n = ha.hattn_prefill_backward_workspace_size(32768, 64, 8)
    assert n == 32768 * 64 * 128 + 32768 * 8 * 128 + 32768 * 64 * 4 + 1024 * 64 * 4
    r = lambda x: (x + 255) // 256 * 256
    assert ha.hattn_prefill_backward_workspace_size(33, 4, 2) == \
        r(33 * 4 * 128) + r(33 * 2 * 128) + r(33 * 4 * 4) + r(2 * 4 * 4)
    assert ha.hattn_prefill_backward_workspace_size(0, 4, 2) == 0


def _backward(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, sink=FAKE, out=FAKE, lse=FAKE, dout=FAKE, grad_q=FAKE,
                grad_k=FAKE, grad_v=FAKE, grad_sink=FAKE, batch=1, cu_seqlens=FAKE,
                total_tokens=512, max_seqlen=512, hq=8, hkv=1, dqk=192, dv=128, rope_dim=64,
                rope_base=1e4, window=128, softmax_scale=0.07, workspace=FAKE,
                workspace_bytes=1 << 24, stream=0)
    args.update(kw)
    return ha.hattn_prefill_backward(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(hkv=3), ha.HATTN_ERR_INVALID_ARG),
    (dict(dqk=128), ha.HATTN_ERR_UNSUPPORTED),
    (dict(hq=64, hkv=2), ha.HATTN_ERR_UNSUPPORTED),      # G = 32
    (dict(lse=None), ha.HATTN_ERR_INVALID_ARG),           # the backward needs the forward's lse
    (dict(dout=None), ha.HATTN_ERR_INVALID_ARG),
    (dict(grad_sink=None), ha.HATTN_ERR_INVALID_ARG),
    (dict(grad_q=FAKE + 8), ha.HATTN_ERR_INVALID_ARG),    # misaligned
    (dict(dout=FAKE + 2), ha.HATTN_ERR_INVALID_ARG),
    (dict(window=-1), ha.HATTN_ERR_INVALID_ARG),
    (dict(softmax_scale=float("inf")), ha.HATTN_ERR_INVALID_ARG),
    (dict(max_seqlen=513), ha.HATTN_ERR_INVALID_ARG),
    (dict(workspace_bytes=1000), ha.HATTN_ERR_WORKSPACE),
    (dict(workspace=None), ha.HATTN_ERR_WORKSPACE),
    (dict(batch=0), ha.HATTN_ERR_INVALID_ARG),
])
def test_backward_rejects_bad_arguments(lib, kw, code):
    assert _backward(**kw) == code


def test_injected_launch_failures_are_consumed_by_launching_calls(lib):
    """Host-side fault injection: pending failures are consumed only by calls
    that passed their argument checks, each returning HATTN_ERR_CUDA."""
    assert ha.hattn_test_fail_next_launches(2) == 0
    try:
        assert _prefill(hkv=3) == ha.HATTN_ERR_INVALID_ARG       # rejected first: not consumed
        assert _decode(cap=130) == ha.HATTN_ERR_RING_TOO_SMALL
        assert ha.hattn_test_fail_next_launches(2) == 2
        assert _prefill(workspace_bytes=1 << 20) == ha.HATTN_ERR_CUDA
        assert ha.hattn_test_fail_next_launches(2) == 1
        assert _decode() == ha.HATTN_ERR_CUDA
        assert _backward() == ha.HATTN_ERR_CUDA
        assert ha.hattn_test_fail_next_launches(0) == 0
    finally:
        ha.hattn_test_fail_next_launches(0)
