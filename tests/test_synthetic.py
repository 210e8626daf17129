"""The seeded input generators: determinism and the structural promises the
tests and the bench rely on (they compute no part of the attention)."""

import numpy as np

from paged_decode_attention_fp8_gb300 import synthetic as syn


def test_affine_index_rule_gives_distinct_rows_in_range():
    a = syn.sparse_inputs(7, 64, num_tokens=4096, topk=256, index_rule="affine")
    b = syn.sparse_inputs(7, 64, num_tokens=4096, topk=256, index_rule="affine")
    idx = a.topk_idx.numpy()
    assert idx.shape == (64, 256)
    assert np.array_equal(idx, b.topk_idx.numpy())                  # seeded
    assert idx.min() >= 0 and idx.max() < 4096
    assert all(len(np.unique(r)) == 256 for r in idx)               # top-k rows are distinct
    assert len({tuple(r[:8]) for r in idx}) == 64                   # tokens differ


def test_permutation_rule_is_the_default_and_distinct():
    a = syn.sparse_inputs(7, 3, num_tokens=4096, topk=256)
    b = syn.sparse_inputs(7, 3, num_tokens=4096, topk=256, index_rule="permutation")
    assert np.array_equal(a.topk_idx.numpy(), b.topk_idx.numpy())
    assert all(len(np.unique(r)) == 256 for r in a.topk_idx.numpy())


def test_cache_write_slots_are_distinct_and_follow_pages():
    inp = syn.cache_write_inputs(8, [17, 40, 1], page=16, spare_blocks=2, pad_tokens=3)
    s = inp.slot_mapping.numpy()
    real = s[s >= 0]
    assert len(s) == 17 + 40 + 1 + 3 and len(real) == 58
    assert len(np.unique(real)) == len(real) and real.max() < inp.num_blocks * 16
    # consecutive tokens of a sequence share a block until the page fills
    first = real[:17]
    assert np.all(first[:16] // 16 == first[0] // 16) and np.all(first % 16 == np.arange(17) % 16)
