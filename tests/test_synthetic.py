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


def _decoded(codes):
    from oracle.attention import e4m3_decode  # the oracle's table, used here only to read bytes back
    return e4m3_decode(codes)


def test_pooled_mla_values_keep_the_scale_rule_and_the_poison():
    sl = [8196, 100, 5, 700, 0]
    inp = syn.mla_inputs(3, len(sl), 2, 64, sl, causal=True, spare_pages=2, value_pages=8)
    cache, bt = inp.kv_cache.numpy(), inp.block_table.numpy()
    valid = []
    for i, s_k in enumerate(sl):
        for p in range((s_k + 63) // 64):
            rows = cache[bt[i, p]]
            n = min(64, s_k - 64 * p)
            valid.append(rows[:n])
            assert np.all(rows[n:] == syn.POISON_BYTE)
    v = _decoded(np.concatenate(valid))
    assert np.all(np.isfinite(v))
    assert np.max(np.abs(v)) == 448.0       # amax / 448 over the valid rows: the largest encodes to 448
    # seeded, and the pool is shared between pages (bounded distinct values)
    again = syn.mla_inputs(3, len(sl), 2, 64, sl, causal=True, spare_pages=2, value_pages=8)
    assert np.array_equal(cache, again.kv_cache.numpy())


def test_pooled_gqa_values_keep_the_scale_rule_and_the_poison():
    sl = [1024, 17, 300]
    inp = syn.gqa_inputs(5, 3, sl, spare_blocks=2, value_blocks=4)
    for cache in (inp.k_cache.numpy(), inp.v_cache.numpy()):
        bt = inp.block_table.numpy()
        valid = []
        for i, s_k in enumerate(sl):
            for p in range((s_k + 15) // 16):
                blk = cache[bt[i, p]]
                n = min(16, s_k - 16 * p)
                valid.append(blk[:, :n].reshape(-1, 128))
                assert np.all(blk[:, n:] == syn.POISON_BYTE)
        v = _decoded(np.concatenate(valid))
        assert np.all(np.isfinite(v)) and np.max(np.abs(v)) == 448.0
