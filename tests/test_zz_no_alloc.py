"""fp8mla_decode_no_alloc: the dense MLA decode for callers that cannot
allocate device memory, checked against fp8mla_decode on the same inputs.

Such callers pass only inputs and outputs; the library keeps the schedule and
the LSE-correction terms in a fixed array of its own.  Two different batches
are decoded in a row, so the second call runs on whatever the first one left
in that array.  fp8mla_decode runs with one unit per sequence too
(force_splits=1), the schedule the no-allocation variant uses.
"""

import pytest
import torch

import paged_decode_attention_fp8_gb300 as fm
from paged_decode_attention_fp8_gb300 import synthetic as syn
from tests.parity import TOL

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
def test_no_alloc_matches_decode_on_two_calls_in_a_row(mode):
    batches = [syn.mla_inputs(31, 6, 2, 64, [700, 1, 2048, 0, 130, 4000], causal=True, spare_pages=4),
               syn.mla_inputs(32, 3, 1, 16, [256, 300, 64], causal=False, spare_pages=2)]
    for inp in batches:
        d = _dev(inp)
        ref_out, ref_lse = _existing(inp, d, mode)
        out, lse = fm.decode_no_alloc(d["q"], d["kv"], d["bt"], d["sl"], d["scale"], inp.softmax_scale,
                                      inp.causal, dot_mode=mode)
        torch.cuda.synchronize()
        rel = ((out.float() - ref_out.float()).norm() / ref_out.float().norm()).item()
        finite = torch.isfinite(ref_lse)
        assert torch.equal(torch.isfinite(lse), finite)
        assert rel <= TOL[mode]["rel_l2"]
        assert (lse[finite] - ref_lse[finite]).abs().max().item() <= TOL[mode]["lse"]
        assert fm.last_device_error() == 0


def test_no_alloc_refuses_a_batch_beyond_its_array():
    inp = syn.mla_inputs(33, fm.NO_ALLOC_MAX_BATCH + 1, 1, 16, [64] * (fm.NO_ALLOC_MAX_BATCH + 1), causal=False)
    d = _dev(inp)
    with pytest.raises(fm.FP8MLAError) as err:
        fm.decode_no_alloc(d["q"], d["kv"], d["bt"], d["sl"], d["scale"], inp.softmax_scale, False)
    assert err.value.status == 3
