"""Bounded waits of the dense FP8-dots MLA decode, exercised without a GPU fault.

The library's test hook makes one CTA skip the loads of one page, so the
waits on that page (and, once that CTA stops, its peers' waits) can only end
by running out.  The decode must return with FP8MLA_DEV_WAIT_TIMEOUT recorded
and the source line of the first wait that gave up, and the CUDA context must
stay usable: the next decode, with the hook off, matches the oracle and
reproduces the run made before the fault.
"""

import pytest
import torch

import oracle
import paged_decode_attention_fp8_gb300 as fm
from paged_decode_attention_fp8_gb300 import synthetic as syn
from tests.parity import assert_close, compare

pytestmark = pytest.mark.gpu

LIMIT_NS = 20_000_000  # 20 ms: long enough for any live wait here, short enough for a fast test


def _inputs():
    inp = syn.mla_inputs(5, 2, 2, 64, [700, 389], causal=True, spare_pages=8)
    dev = torch.device("cuda")
    d = dict(q=inp.q.to(dev), kv=inp.kv_cache.to(dev), bt=inp.block_table.to(dev), sl=inp.seqlens.to(dev),
             scale=torch.tensor([inp.kv_scale], dtype=torch.float32, device=dev))
    return inp, d


def _decode(inp, d, units):
    ts, ns = fm.get_metadata(d["sl"], inp.h_q, inp.s_q, num_units=units)
    out, lse = fm.decode(d["q"], d["kv"], d["bt"], d["sl"], d["scale"], inp.softmax_scale, inp.causal, ts, ns,
                         dot_mode="fp8")
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("fault_page", [1, 3])
def test_wait_runs_out_and_context_survives(fault_page):
    inp, d = _inputs()
    units = 1  # one unit holds every page, so unit 0 sees the skipped page
    fm.last_device_error()
    fm.wait_timeout_site()
    before_out, before_lse = _decode(inp, d, units)
    assert fm.last_device_error() == 0
    try:
        fm.set_wait_test(fault_page, LIMIT_NS)
        _decode(inp, d, units)
        code = fm.last_device_error()
        site = fm.wait_timeout_site()
    finally:
        fm.set_wait_test(0, 0)
    assert code & fm.DEV_WAIT_TIMEOUT, f"status {code:#x}"
    assert site is not None and site[0] > 0, site
    # the context is usable: the same call again is correct and reproduces the run before the fault
    out, lse = _decode(inp, d, units)
    assert fm.last_device_error() == 0
    assert fm.wait_timeout_site() is None
    assert torch.equal(out, before_out) and torch.equal(lse, before_lse)
    ro, rl = oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens, inp.kv_scale,
                               inp.softmax_scale, inp.causal)
    assert_close(compare(out, lse, ro, rl, "fp8"), "fp8")


def test_hook_rejects_negative_page():
    with pytest.raises(fm.FP8MLAError):
        fm.set_wait_test(-1, 0)
