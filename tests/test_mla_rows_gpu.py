"""Dense MLA decode with one KV scale per cached row (fp8mla_decode_ext, FP8
dots) on the GPU against the fp64 oracle.

The InfiniCore FP8 paged-attention page (Summary) keeps scales of shape
[num_blocks, num_kv_heads, block_size]; the dense MLA cache has one KV head,
so [num_pages, 1, 64], and a row's scale applies to its latent part (K and V)
and its RoPE part alike.  Checked with seeded scales over ragged lengths,
forced splits and the MTP shape, and end to end after the library's own
quantise-on-write filled an MLA-layout cache and its scales.

The keys keep N(0, 1) statistics while their scales span a factor of 8, so the
FP8-dot tolerance of the per-tensor tests applies unchanged: the kernel rounds
Q to E4M3, and keys several times larger than that would sharpen the softmax
and grow the second-order part of that rounding's LSE error, which the
per-tensor tests do not allow for either.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_fp8_gb300 as fm
from paged_decode_attention_fp8_gb300 import synthetic as syn
from tests.parity import assert_close, compare

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _run(inp, rows, force_splits=0, units=None, q=None):
    d = dict(q=(inp.q if q is None else q).to(DEV), kv=inp.kv_cache.to(DEV), bt=inp.block_table.to(DEV),
             sl=inp.seqlens.to(DEV))
    ts, ns = fm.get_metadata(d["sl"], inp.h_q, inp.s_q, num_units=units, force_splits=force_splits)
    out, lse = fm.decode(d["q"], d["kv"], d["bt"], d["sl"], rows.to(DEV), inp.softmax_scale, inp.causal, ts, ns,
                         dot_mode="fp8")
    torch.cuda.synchronize()
    return out, lse


CASES = [  # (b, s_q, h_q, seqlens, force_splits)
    (4, 2, 64, [700, 1, 2048, 0], 0),
    (4, 2, 64, [700, 65, 2048, 333], 3),
    (3, 1, 16, [256, 300, 64], 1),
]


@pytest.mark.parametrize("case", CASES, ids=[f"b{c[0]}_sq{c[1]}_h{c[2]}_fs{c[4]}" for c in CASES])
def test_per_row_scales_match_oracle(case):
    b, s_q, h_q, seqlens, fs = case
    inp, rows = syn.mla_row_scaled_inputs(61, b, s_q, h_q, seqlens, causal=True, spare_pages=3)
    out, lse = _run(inp, rows, force_splits=fs)
    ro, rl = oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens, rows.numpy(), inp.softmax_scale,
                               inp.causal)
    assert_close(compare(out, lse, ro, rl, "fp8"), "fp8")
    assert fm.last_device_error() == 0


def test_per_row_scales_mtp_shape_sampled():
    """b = 64, s_q = 2, h_q = 64 at the MTP lengths, 6 sequences checked against the oracle."""
    seqlens = syn.uniform_seqlens(2, 64, 2048, 6144)
    inp, rows = syn.mla_row_scaled_inputs(62, 64, 2, 64, seqlens, causal=True, spare_pages=8, value_pages=96)
    out, lse = _run(inp, rows)
    pick = [0, 9, 17, 33, 48, 63]
    ro, rl = oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens, rows.numpy(), inp.softmax_scale,
                               inp.causal, batches=pick)
    m = np.zeros(64, dtype=bool)
    m[pick] = True
    assert_close(compare(out, lse, ro, rl, "fp8", mask=m), "fp8")
    assert fm.last_device_error() == 0


def test_uniform_rows_equal_per_tensor():
    """Every row scale equal to the tensor scale: the same result as the per-tensor call, within
    the FP8-dot tolerance (the two paths round P against different references)."""
    inp = syn.mla_inputs(63, 3, 2, 64, [900, 130, 64], causal=True, spare_pages=2)
    rows = torch.full((inp.kv_cache.shape[0], 1, 64), inp.kv_scale, dtype=torch.float32)
    out_r, lse_r = _run(inp, rows)
    out_t, lse_t = _run(inp, torch.tensor([inp.kv_scale], dtype=torch.float32))
    m = compare(out_r, lse_r, out_t.float().cpu().numpy().astype(np.float64), lse_t.cpu().numpy(), "fp8")
    assert_close(m, "fp8")


def test_write_then_decode_round_trip():
    """An MLA-layout cache and its per-row scales written by fp8_paged_cache_write, then decoded:
    the decode matches the oracle on exactly the bytes and scales that were written."""
    seqlens = [517, 64, 1300, 33]
    wi = syn.cache_write_inputs(64, seqlens, h_kv=1, hd=576, page=64, base_tokens=512, spare_blocks=2,
                                exp_range=0)
    x = syn.materialise(wi)
    n = wi.num_blocks
    cache = torch.zeros((n, 1, 64, 576), dtype=torch.uint8, device=DEV)
    scales = torch.ones((n, 1, 64), dtype=torch.float32, device=DEV)
    fm.paged_cache_write(x.to(DEV), wi.slot_mapping.to(DEV), cache, token_scales=scales)
    torch.cuda.synchronize()
    assert fm.last_device_error() == 0
    slots = wi.slot_mapping.numpy()
    max_pages = max((s + 63) // 64 for s in seqlens)
    bt = np.zeros((len(seqlens), max_pages), dtype=np.int32)
    t = 0
    for i, s in enumerate(seqlens):
        for p in range((s + 63) // 64):
            bt[i, p] = slots[t + 64 * p] // 64
        t += s
    q = syn.to_bf16(syn.normal(64, 72, (len(seqlens), 2, 64, 576)))
    kv = cache.view(n, 64, 576)
    bt_t, sl = torch.from_numpy(bt), torch.tensor(seqlens, dtype=torch.int32)
    ts, ns = fm.get_metadata(sl.to(DEV), 64, 2)
    softmax_scale = 576 ** -0.5
    out, lse = fm.decode(q.to(DEV), kv, bt_t.to(DEV), sl.to(DEV), scales, softmax_scale, True, ts, ns,
                         dot_mode="fp8")
    torch.cuda.synchronize()
    ro, rl = oracle.mla_decode(q, kv.cpu(), bt_t, sl, scales.cpu().numpy(), softmax_scale, True)
    assert_close(compare(out, lse, ro, rl, "fp8"), "fp8")
    assert fm.last_device_error() == 0
