"""The kernels' barrier protocols under random schedules (tests/protocol_model.py).

Each protocol runs over a few hundred random interleavings of its roles, TMA
copies and tensor-core products; none may take an arrival beyond a barrier's
count, read a buffer's wrong contents or deadlock.  Planted mistakes --
protocols that an earlier version of the kernels had, or that the staging of
O would have without its waits -- must be caught, which shows the models can
fail.
"""
import random

import pytest

import protocol_model as pm

MIXES = [[1] * 7, [1, 1, 2, 1, 3, 1, 1], [3, 1, 1, 2], [2] * 5, [5, 1, 1, 1, 4]]


def _random_mixes(n, seed, choices, lo, hi):
    rs = random.Random(seed)
    return [[rs.choice(choices) for _ in range(rs.randint(lo, hi))] for _ in range(n)]


@pytest.mark.parametrize("kst", [2, 3])
def test_multi_block_prefill_protocol(kst):
    for units in MIXES + _random_mixes(20, kst, [1, 1, 2, 3, 5], 3, 9):
        for seed in range(15):
            pm.multi_block_prefill(units, seed, kst=kst)


def test_multi_block_prefill_catches_one_k0_barrier_for_all_units():
    # one K_0 barrier for every unit: with one-block units the producer can
    # issue the next unit's K_0 before the last one has landed
    failures = 0
    for seed in range(60):
        try:
            pm.multi_block_prefill([1] * 7, seed, shared_k0_barrier=True)
        except RuntimeError as e:  # a second arrival in one phase, or a wait that aliased
            assert any(w in str(e) for w in ("too many arrivals", "reads", "deadlock")), e
            failures += 1
    assert failures > 0


@pytest.mark.parametrize("nunits", [1, 2, 3, 6])
def test_one_block_prefill_protocol(nunits):
    for seed in range(150):
        pm.one_block_prefill(nunits, seed)


@pytest.mark.parametrize("mistake", ["stage_a_after_own_pv", "v_without_o_read"])
def test_one_block_prefill_catches_staging_mistakes(mistake):
    # tile A staging O into the V stage before PV_B has read it, or the next
    # V block loaded before the staged O has been read out
    failures = 0
    for seed in range(200):
        try:
            pm.one_block_prefill(4, seed, **{mistake: True})
        except (AssertionError, RuntimeError):
            failures += 1
    assert failures > 0


def test_split_kv_decode_protocol():
    for items in _random_mixes(40, 11, [1, 1, 2, 3, 4, 7], 2, 8):
        for seed in range(10):
            pm.split_kv_decode(items, seed)


def test_split_kv_decode_catches_epilogue_on_pv_done_parity():
    # the epilogue waiting on the per-block PV barrier with the parity of the
    # item's last block: the row warps get there having seen only the PVs up
    # to two blocks back, so the parity can already read complete
    failures = 0
    for seed in range(80):
        try:
            pm.split_kv_decode([7, 2, 7, 4], seed, epilogue_on_pv_done=True)
        except (AssertionError, RuntimeError):
            failures += 1
    assert failures > 0


@pytest.mark.parametrize("entries", [1, 3, 4, 9, 30])
def test_unit_queue_protocol(entries):
    # the MMA issuer and the eight softmax warps read every entry once, in
    # order, whatever their lead or lag
    for seed in range(40):
        pm.unit_queue(entries, 9, seed)


def test_unit_queue_catches_slot_reuse_before_all_read():
    failures = 0
    for seed in range(60):
        try:
            pm.unit_queue(12, 9, seed, skip_empty_wait=True)
        except RuntimeError:
            failures += 1
    assert failures > 0
