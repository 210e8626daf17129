"""Top-k sparse MLA decode on the GPU against the fp64 oracle (through the C ABI).

Shapes follow the aiter sparse_mla_fwd page (Results): 16 heads, rope-free
d = dv = 512, one E4M3 cache of 131072 tokens, top-k 2048 distinct indices,
decode with 2 and 16 query tokens, FP8 Q/P dots; plus its Accuracy case --
one key +9 above 2047 that carry a fifth of the output, split-K off.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_fp8_gb300 as fm
from paged_decode_attention_fp8_gb300 import synthetic as syn
from tests.parity import assert_close, compare, record

pytestmark = pytest.mark.gpu


def run(inp, num_splits=0, idx=None):
    dev = torch.device("cuda")
    idx = inp.topk_idx if idx is None else idx
    scale = torch.tensor([inp.kv_scale], dtype=torch.float32, device=dev)
    out, lse = fm.sparse_mla_decode(inp.q.to(dev), inp.kv_cache.to(dev), idx.to(dev), scale,
                                    inp.softmax_scale, num_splits=num_splits)
    torch.cuda.synchronize()
    return out, lse


def ref(inp, idx=None):
    return oracle.sparse_mla_decode(inp.q, inp.kv_cache, inp.topk_idx if idx is None else idx,
                                    inp.kv_scale, inp.softmax_scale)


@pytest.mark.parametrize("s_q", [2, 16])
@pytest.mark.parametrize("splits", [0, 1, 4])
def test_decode_shapes(s_q, splits):
    inp = syn.sparse_inputs(4, s_q)
    out, lse = run(inp, splits)
    ro, rl = ref(inp)
    m = compare(out, lse, ro, rl, "fp8")
    record(f"sparse_sq{s_q}_splits{splits}", m)
    assert_close(m, "fp8")
    assert fm.last_device_error() == 0


def test_peaky_tail_kept_with_split_off():
    inp = syn.sparse_peaky_inputs(4, s_q=2)
    out, lse = run(inp, num_splits=1)
    ro, rl = ref(inp)
    m = compare(out, lse, ro, rl, "fp8")
    record("sparse_peaky_splits1", m)
    assert_close(m, "fp8")
    # the value dims [256, 512) carry 0.8 z + 0.2 w: a lost tail moves them by ~20%
    mv = compare(out[..., 256:], lse, ro[..., 256:], rl, "fp8")
    record("sparse_peaky_value_dims", mv)
    assert mv["rel_l2"] < 5e-2


def test_skipped_and_ragged_indices():
    inp = syn.sparse_inputs(9, 3, h_q=16, num_tokens=5000, topk=300)
    idx = inp.topk_idx.clone()
    idx[0, ::3] = -1          # some keys skipped
    idx[1, :] = -1            # a token with no key at all
    idx[2, 10:20] = idx[2, 0]  # repeated rows count once per listing
    for splits in (1, 2, 0):
        out, lse = run(inp, splits, idx)
        ro, rl = ref(inp, idx)
        m = compare(out, lse, ro, rl, "fp8")
        assert_close(m, "fp8")
    assert fm.last_device_error() == 0


@pytest.mark.parametrize("splits", [2, 3, 5, 8, 9, 16])
def test_split_counts(splits):
    # every split count up to one per 128-key chunk, counts that do not
    # divide the 16 chunks evenly included
    inp = syn.sparse_inputs(14, 2)
    out, lse = run(inp, num_splits=splits)
    ro, rl = ref(inp)
    m = compare(out, lse, ro, rl, "fp8")
    record(f"sparse_sq2_splits{splits}_counts", m)
    assert_close(m, "fp8")
    assert fm.last_device_error() == 0


def test_split_merge_empty_shards_and_fewer_heads():
    # 4 splits where one token has no key at all and another has keys in its
    # first shard only, with 5 heads
    inp = syn.sparse_inputs(15, 3, h_q=5, num_tokens=6000, topk=512)
    idx = inp.topk_idx.clone()
    idx[0, :] = -1
    idx[1, 128:] = -1
    out, lse = run(inp, num_splits=4, idx=idx)
    ro, rl = ref(inp, idx)
    assert_close(compare(out, lse, ro, rl, "fp8"), "fp8")
    assert fm.last_device_error() == 0


@pytest.mark.parametrize("s_q,splits", [(38, 4), (48, 4), (3, 24)])
def test_split_merge_more_tokens_and_many_splits(s_q, splits):
    # more CTAs than SMs (48 x 4), and more than 16 splits per token (the
    # combine kernel's general path: a CTA-wide maximum, then 16 splits at a time)
    inp = syn.sparse_inputs(13, s_q, num_tokens=8192, topk=3072)
    out, lse = run(inp, num_splits=splits)
    ro, rl = ref(inp)
    assert_close(compare(out, lse, ro, rl, "fp8"), "fp8")
    assert fm.last_device_error() == 0


def test_fewer_heads():
    inp = syn.sparse_inputs(10, 2, h_q=5, num_tokens=4096, topk=512)
    out, lse = run(inp)
    ro, rl = ref(inp)
    assert_close(compare(out, lse, ro, rl, "fp8"), "fp8")


def test_run_to_run_bit_identical():
    inp = syn.sparse_inputs(11, 2, num_tokens=8192, topk=1024)
    a = run(inp)
    b = run(inp)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_out_of_range_index_reported():
    inp = syn.sparse_inputs(12, 1, num_tokens=1024, topk=256)
    idx = inp.topk_idx.clone()
    idx[0, 5] = 5000
    run(inp, 1, idx)
    assert fm.last_device_error() & fm.DEV_BAD_INDEX


def test_prefill_scale_sampled():
    # the aiter page's prefill leg: 16 384 query tokens, 16 heads, top-k 2048
    # over a 131 072-token E4M3 cache (indices by the affine rule); the whole
    # batch runs with the automatic split choice, 24 tokens spread over it
    # are checked against the oracle one by one
    inp = syn.sparse_inputs(4, 16384, index_rule="affine")
    assert fm.sparse_workspace_bytes(16384, 16, 2048, 0) < (1 << 30)
    out, lse = run(inp, num_splits=0)
    picks = sorted({int(x) for x in np.linspace(0, 16383, 24)})
    ro, rl = oracle.sparse_mla_decode(inp.q, inp.kv_cache, inp.topk_idx, inp.kv_scale, inp.softmax_scale,
                                      tokens=picks)
    m = compare(out[picks], lse[picks], ro[picks], rl[picks], "fp8")
    record("sparse_prefill_sq16384_sampled", m)
    assert_close(m, "fp8")
    assert fm.last_device_error() == 0


def test_alternating_caches_use_their_own_tensor_maps():
    # the entry point keeps encoded tensor maps by (base pointer, extent, device): calls that
    # alternate between two caches of one shape, and a third of another size, each read their own
    a = syn.sparse_inputs(16, 2, num_tokens=4096, topk=512)
    b = syn.sparse_inputs(17, 2, num_tokens=4096, topk=512)
    c = syn.sparse_inputs(18, 2, num_tokens=6000, topk=512)
    for inp in (a, b, a, c, b):
        out, lse = run(inp)
        ro, rl = ref(inp)
        assert_close(compare(out, lse, ro, rl, "fp8"), "fp8")
    assert fm.last_device_error() == 0
