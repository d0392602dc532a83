"""Pins of the ragged multi-user decode plan (integer work list), CPU only."""
import math

import pytest

import oracle


def test_closed_forms():
    # nothing attended: the minimum chunk and no work
    assert oracle.varlen_plan([0, 0], 4096, 8, 253) == (512, [])
    # 1000 keys, 8 KV heads, target 253: ceil(8000 / 253) = 32 -> 64 -> min 512
    assert oracle.varlen_plan([1000], 1000, 8, 253) == (512, [(0, 0, 512), (0, 512, 1000)])
    # one 128K user and 31 users of 2K: T = 194560, ceil(T * 8 / 253) = 6153 -> 6208
    c, items = oracle.varlen_plan([131072] + [2048] * 31, 131072, 8, 253)
    assert c == 6208
    assert sum(1 for b, _, _ in items if b == 0) == math.ceil(131072 / 6208)
    assert all(hi - lo == 2048 for b, lo, hi in items if b > 0)
    # lengths are clamped to [0, max_seqlen]
    assert oracle.varlen_plan([-5, 9999], 600, 1, 1000) == (512, [(1, 0, 512), (1, 512, 600)])


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("hkv,target", [(8, 253), (1, 253), (2, 40), (16, 500)])
def test_chunks_partition_each_sequence_and_fit_the_capacity(seed, hkv, target):
    import random
    rnd = random.Random(seed)
    B = rnd.randint(1, 40)
    s_max = rnd.choice([64, 1000, 32768, 131072])
    lens = [rnd.choice([0, 1, rnd.randint(0, s_max), s_max]) for _ in range(B)]
    c, items = oracle.varlen_plan(lens, s_max, hkv, target)
    assert c % 64 == 0 and c >= 512
    assert len(items) <= -(-target // hkv) + B  # the capacity the workspace reserves
    for b in range(B):
        mine = [(lo, hi) for bb, lo, hi in items if bb == b]
        pos = 0
        for lo, hi in mine:  # contiguous, in order, each at most C keys
            assert lo == pos and 0 < hi - lo <= c
            pos = hi
        assert pos == min(lens[b], s_max)
    assert [b for b, _, _ in items] == sorted(b for b, _, _ in items)
