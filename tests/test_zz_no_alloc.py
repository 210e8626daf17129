"""fp8mla_decode_no_alloc: the dense MLA decode for callers that cannot
allocate device memory.

Such callers pass only inputs and outputs; the library keeps the tile
schedule, the split counts and the quantised Q (its E4M3 hi term, in both dot
modes) with its per-row scales in a fixed device array of its own.  It
schedules one unit per sequence, so fp8mla_decode with one unit per sequence
(force_splits=1) runs the same kernels on the same schedule: the results must
be bit-identical.  Two different batches are decoded in a row, so the second
call runs on whatever the first one left in that array, and a batch of
FP8MLA_NO_ALLOC_MAX_BATCH sequences (whose per-row scales end on the array's
last byte) is checked against the oracle in both dot modes.
"""

import pytest
import torch

import oracle
import paged_decode_attention_fp8_gb300 as fm
from paged_decode_attention_fp8_gb300 import synthetic as syn
from tests.parity import assert_close, compare

pytestmark = pytest.mark.gpu


def _existing(inp, d, mode):
    ts, ns = fm.get_metadata(d["sl"], inp.h_q, inp.s_q, num_units=inp.b, force_splits=1)
    return fm.decode(d["q"], d["kv"], d["bt"], d["sl"], d["scale"], inp.softmax_scale, inp.causal, ts, ns,
                     dot_mode=mode)


def _dev(inp):
    dev = torch.device("cuda")
    return dict(q=inp.q.to(dev), kv=inp.kv_cache.to(dev), bt=inp.block_table.to(dev), sl=inp.seqlens.to(dev),
                scale=torch.tensor([inp.kv_scale], dtype=torch.float32, device=dev))


@pytest.mark.parametrize("mode", ["fp8", "bf16"])
def test_no_alloc_bit_identical_to_decode_on_two_calls_in_a_row(mode):
    batches = [syn.mla_inputs(31, 6, 2, 64, [700, 1, 2048, 0, 130, 4000], causal=True, spare_pages=4),
               syn.mla_inputs(32, 3, 1, 16, [256, 300, 64], causal=False, spare_pages=2)]
    for inp in batches:
        d = _dev(inp)
        ref_out, ref_lse = _existing(inp, d, mode)
        out, lse = fm.decode_no_alloc(d["q"], d["kv"], d["bt"], d["sl"], d["scale"], inp.softmax_scale,
                                      inp.causal, dot_mode=mode)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out)
        assert torch.equal(lse.isnan(), ref_lse.isnan())
        assert torch.equal(lse.nan_to_num(0.0), ref_lse.nan_to_num(0.0))
        assert fm.last_device_error() == 0


@pytest.mark.parametrize("mode", ["fp8", "bf16"])
def test_no_alloc_full_array_matches_oracle(mode):
    b = fm.NO_ALLOC_MAX_BATCH
    seqlens = [(37 * i) % 300 + (i % 3) for i in range(b)]  # short caches, a few empty ones
    inp = syn.mla_inputs(34, b, 2, 64, seqlens, causal=True, spare_pages=4)
    d = _dev(inp)
    out, lse = fm.decode_no_alloc(d["q"], d["kv"], d["bt"], d["sl"], d["scale"], inp.softmax_scale, inp.causal,
                                  dot_mode=mode)
    torch.cuda.synchronize()
    assert fm.last_device_error() == 0
    ro, rl = oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens, inp.kv_scale,
                               inp.softmax_scale, inp.causal)
    assert_close(compare(out, lse, ro, rl, mode), mode)
    ref_out, ref_lse = _existing(inp, d, mode)
    assert torch.equal(out, ref_out)


def test_no_alloc_refuses_a_batch_beyond_its_array():
    inp = syn.mla_inputs(33, fm.NO_ALLOC_MAX_BATCH + 1, 1, 16, [64] * (fm.NO_ALLOC_MAX_BATCH + 1), causal=False)
    d = _dev(inp)
    with pytest.raises(fm.FP8MLAError) as err:
        fm.decode_no_alloc(d["q"], d["kv"], d["bt"], d["sl"], d["scale"], inp.softmax_scale, False)
    assert err.value.status == 3
