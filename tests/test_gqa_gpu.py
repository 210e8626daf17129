"""Paged GQA decode on the GPU against the fp64 oracle (through the C ABI).

Shapes follow the InfiniCore FP8 paged-attention page: 32 query heads, 8 KV
heads, head_dim 128, page 16, separate E4M3 K and V with per-tensor scales;
bs=1 at context 1024 and 16384, bs=32 with contexts uniform in
[1024, 16384]; split-KV auto and forced to 1, 4 and 8.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_fp8_gb300 as fm
from paged_decode_attention_fp8_gb300 import synthetic as syn
from tests.parity import assert_close, compare, record

pytestmark = pytest.mark.gpu


def run(inp, num_splits=0):
    dev = torch.device("cuda")
    ks = torch.tensor([inp.k_scale], dtype=torch.float32, device=dev)
    vs = torch.tensor([inp.v_scale], dtype=torch.float32, device=dev)
    out, lse = fm.paged_gqa_decode(inp.q.to(dev), inp.k_cache.to(dev), inp.v_cache.to(dev),
                                   inp.block_table.to(dev), inp.seqlens.to(dev), ks, vs,
                                   inp.softmax_scale, num_splits=num_splits)
    torch.cuda.synchronize()
    return out, lse


def ref(inp):
    return oracle.gqa_decode(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.seqlens,
                             inp.k_scale, inp.v_scale, inp.softmax_scale)


CASES = {
    "bs1_ctx1024": (1, [1024]),
    "bs1_ctx16384": (1, [16384]),
    "bs32_varlen": (32, None),
}


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("splits", [0, 1, 4, 8])
def test_config_cases(case, splits):
    bs, seqlens = CASES[case]
    if seqlens is None:
        seqlens = syn.uniform_seqlens(5, bs, 1024, 16384)
    inp = syn.gqa_inputs(5, bs, seqlens, spare_blocks=16)
    out, lse = run(inp, splits)
    ro, rl = ref(inp)
    m = compare(out, lse, ro, rl, "bf16")
    record(f"gqa_{case}_splits{splits}", m)
    assert_close(m, "bf16")
    assert fm.last_device_error() == 0


@pytest.mark.parametrize("group", [1, 4, 8, 16])
def test_ragged_lengths_and_groups(group):
    seqlens = [0, 1, 15, 16, 17, 127, 128, 129, 300]
    h_kv = 2
    inp = syn.gqa_inputs(6, len(seqlens), seqlens, h_q=h_kv * group, h_kv=h_kv, spare_blocks=4)
    for splits in (1, 3):
        out, lse = run(inp, splits)
        ro, rl = ref(inp)
        assert_close(compare(out, lse, ro, rl, "bf16"), "bf16")


def test_auto_split_rule():
    # a full grid is cut into about six CTAs per SM (pieces of >= 8 steps);
    # a lone sequence is split to fill the GPU
    sms = fm.num_sms()
    assert fm.gqa_num_splits(32, 8, 16384) == min(16, -(-6 * sms // 256))
    assert fm.gqa_num_splits(256, 8, 1024) == 1   # pieces would be shorter than 8 steps
    assert fm.gqa_num_splits(1, 8, 16384) > 1
    assert fm.gqa_num_splits(1, 8, 16384, num_splits=4) == 4
    assert fm.gqa_num_splits(1, 8, 256, num_splits=8) == 2   # capped at the 128-token steps present


def test_run_to_run_bit_identical():
    inp = syn.gqa_inputs(7, 4, [3000, 100, 7000, 1], spare_blocks=8)
    a = run(inp, 4)
    b = run(inp, 4)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_bad_block_reported():
    inp = syn.gqa_inputs(8, 2, [100, 40])
    inp.block_table[0, 1] = 10 ** 6
    run(inp, 1)
    assert fm.last_device_error() & fm.DEV_BAD_PAGE


def test_alternating_caches_use_their_own_tensor_maps():
    # encoded tensor maps are kept by (base pointer, extent, device): alternating K/V caches of
    # one shape, and caches of another pool size, each read their own
    a = syn.gqa_inputs(61, 3, [300, 17, 900], spare_blocks=2)
    b = syn.gqa_inputs(62, 3, [300, 17, 900], spare_blocks=2)
    c = syn.gqa_inputs(63, 3, [64, 1000, 5], spare_blocks=9)
    for inp in (a, b, a, c, b):
        out, lse = run(inp, 0)
        ro, rl = ref(inp)
        assert_close(compare(out, lse, ro, rl, "bf16"), "bf16")
    assert fm.last_device_error() == 0
