"""Properties of the restated page-range scheduler (pins that do not use the GPU).

The partition rule is this library's own (the pages describe split-KV
flash-decoding -- InfiniCore "FP8(E4M3) KV cache support in paged
attention", split-kv commit -- but no scheduler), so it is pinned by what any
correct partition must satisfy: every (sequence, page) is covered exactly
once, in order; split counts and split indices agree with the coverage; the
balanced rule keeps every unit within its share of the cost line; the forced
rule cuts near-equal chunks.
"""

import numpy as np
import pytest

import oracle
from oracle.attention import SCHED_FIXED_COST, unit_segments


def _coverage(sched, seqlens, num_splits):
    n = [(int(s) + 63) // 64 for s in seqlens]
    seen = {}
    order = []
    split_ids = {}
    for u in range(sched.shape[0]):
        for (b, lo, hi, k) in unit_segments(sched[u], seqlens):
            assert k == split_ids.get(b, 0)
            split_ids[b] = k + 1
            for p in range(lo, hi):
                assert (b, p) not in seen
                seen[(b, p)] = u
                order.append((b, p))
    expect = [(b, p) for b in range(len(n)) for p in range(n[b])]
    assert order == expect
    for b in range(len(n)):
        assert num_splits[b + 1] - num_splits[b] == split_ids.get(b, 0)
    return seen


@pytest.mark.parametrize("seed", range(20))
def test_balanced_partition_covers_each_page_once(seed):
    rng = np.random.default_rng(seed)
    b = int(rng.integers(1, 130))
    seqlens = rng.integers(0, 9000, size=b)
    seqlens[rng.random(b) < 0.1] = 0
    units = int(rng.integers(1, 80))
    sched, splits = oracle.schedule(seqlens, units)
    _coverage(sched, seqlens, splits)
    n = [(int(s) + 63) // 64 for s in seqlens]
    total = sum(x + SCHED_FIXED_COST for x in n if x > 0)
    share = -(-total // units)
    for u in range(units):
        segs = unit_segments(sched[u], seqlens)
        pages = sum(hi - lo for (_, lo, hi, _) in segs)
        # a unit's cost interval holds at most `share` positions; only a piece that
        # starts mid-sequence brings a fixed cost from outside its interval
        cost = pages + SCHED_FIXED_COST * len(segs)
        assert pages <= share and cost <= share + SCHED_FIXED_COST


def test_headline_batch_is_balanced():
    from paged_decode_attention_fp8_gb300 import synthetic as syn
    seqlens = syn.uniform_seqlens(2, 64, 2048, 6144)
    units = 76
    sched, splits = oracle.schedule(seqlens, units)
    _coverage(sched, seqlens, splits)
    costs = [sum(hi - lo + SCHED_FIXED_COST for (_, lo, hi, _) in unit_segments(sched[u], seqlens))
             for u in range(units)]
    assert max(costs) <= 1.15 * (sum(costs) / units) + SCHED_FIXED_COST


@pytest.mark.parametrize("k", [1, 2, 3, 8])
def test_forced_splits(k):
    seqlens = np.array([256, 300, 0, 1, 64 * 9])
    units = 40
    sched, splits = oracle.schedule(seqlens, units, force_splits=k)
    _coverage(sched, seqlens, splits)
    for b, s in enumerate(seqlens):
        n = (int(s) + 63) // 64
        assert splits[b + 1] - splits[b] == min(k, n)
    sizes = {}
    for u in range(units):
        for (b, lo, hi, _) in unit_segments(sched[u], seqlens):
            sizes.setdefault(b, []).append(hi - lo)
    for b, sz in sizes.items():
        assert max(sz) - min(sz) <= 1


def test_all_empty_batch():
    sched, splits = oracle.schedule([0, 0, 0], 5)
    assert np.all(splits == 0)
    for u in range(5):
        assert unit_segments(sched[u], [0, 0, 0]) == []


def test_balanced_rule_worked_by_hand():
    # pages [10, 3] (64-token pages), 3 units, fixed cost 4 per sequence:
    # cost line 14 + 7 = 21 positions; units start at floor(u * 21 / 3) = 0, 7, 14.
    # position 0 -> sequence 0 page max(0, 0 - 4) = 0; position 7 -> sequence 0 page 3;
    # position 14 -> sequence 1 page 0.  Unit 0 = seq 0 pages [0, 3), unit 1 = seq 0
    # pages [3, 10) (its second piece), unit 2 = seq 1 whole; pieces per sequence 2 and 1.
    sched, ns = oracle.schedule([640, 192], 3)
    assert sched[:, :5].tolist() == [[0, 0, 0, 3, 0], [0, 3, 1, 0, 1], [1, 0, 2, 0, 0]]
    assert ns.tolist() == [0, 2, 3]
    # pages [2, 0, 5], 4 units: cost line 6 + 0 + 9 = 15; units start at positions
    # 0, 3, 7, 11 -> (0, 0); (0, 0) [offset 3 < 4]; (2, 0) [offset 1 of sequence 2];
    # (2, 1) [offset 5, page 5 - 4].  Unit 0 is empty, unit 1 = sequence 0 (sequence 1
    # is empty), unit 2 = sequence 2 page 0, unit 3 = its pages [1, 5) as its second piece.
    sched, ns = oracle.schedule([128, 0, 300], 4)
    assert sched[:, :4].tolist() == [[0, 0, 0, 0], [0, 0, 2, 0], [2, 0, 2, 1], [2, 1, 3, 0]]
    assert ns.tolist() == [0, 1, 1, 3]
