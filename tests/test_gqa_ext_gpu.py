"""Paged GQA decode with per-row KV scales and the XQA options, on the GPU
against the fp64 oracle (through the C ABI, paged_gqa_decode_ext).

Per-row scales follow the InfiniCore FP8 paged-attention page (Summary:
scales [num_blocks, num_kv_heads, block_size]); they are checked with seeded
scales and end to end, after the library's own quantise-on-write produced the
cache and its scales.  The XQA options follow the FlashInfer page "add xqa
fp8 mha and fp8 kv cache" (launcher arguments: a speculative block of q_len
query tokens with its mask, a sliding window, attention sinks; the masked-row
review: a row that sees nothing gives zeros).
"""

import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_fp8_gb300 as fm
from oracle.attention import gqa_decode_ext
from paged_decode_attention_fp8_gb300 import synthetic as syn
from tests.parity import assert_close, compare

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _dev_inputs(inp):
    return dict(kc=inp.k_cache.to(DEV), vc=inp.v_cache.to(DEV), bt=inp.block_table.to(DEV),
                sl=inp.seqlens.to(DEV))


@pytest.mark.parametrize("group", [4, 8])
@pytest.mark.parametrize("splits", [1, 4])
def test_per_row_scales(group, splits):
    h_kv = 2
    inp = syn.gqa_inputs(41, 4, [300, 1, 2000, 777], h_q=h_kv * group, h_kv=h_kv, spare_blocks=6)
    shape = tuple(inp.k_cache.shape[:3])
    ks = syn.per_row_scales(41, 50, shape, inp.k_scale)
    vs = syn.per_row_scales(41, 51, shape, inp.v_scale)
    d = _dev_inputs(inp)
    q = inp.q.unsqueeze(1)  # one query token per sequence
    out, lse = fm.paged_gqa_decode_ext(q.to(DEV), d["kc"], d["vc"], d["bt"], d["sl"], ks.to(DEV), vs.to(DEV),
                                       inp.softmax_scale, num_splits=splits)
    torch.cuda.synchronize()
    ro, rl = oracle.gqa_decode(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.seqlens, ks.numpy(),
                               vs.numpy(), inp.softmax_scale)
    assert_close(compare(out[:, 0], lse[:, 0], ro, rl, "bf16"), "bf16")
    assert fm.last_device_error() == 0


def test_per_tensor_path_unchanged_through_ext():
    """q_len = 1, per-tensor scales, no mask / window / sinks: the same bits as paged_gqa_decode."""
    inp = syn.gqa_inputs(42, 3, [129, 4000, 16], h_q=16, h_kv=4, spare_blocks=3)
    d = _dev_inputs(inp)
    ks = torch.tensor([inp.k_scale], dtype=torch.float32, device=DEV)
    vs = torch.tensor([inp.v_scale], dtype=torch.float32, device=DEV)
    for splits in (1, 3):
        a, la = fm.paged_gqa_decode(inp.q.to(DEV), d["kc"], d["vc"], d["bt"], d["sl"], ks, vs, inp.softmax_scale,
                                    num_splits=splits)
        b, lb = fm.paged_gqa_decode_ext(inp.q.unsqueeze(1).to(DEV), d["kc"], d["vc"], d["bt"], d["sl"], ks, vs,
                                        inp.softmax_scale, num_splits=splits)
        torch.cuda.synchronize()
        assert torch.equal(a, b[:, 0]) and torch.equal(la, lb[:, 0])


def _block_table_from_slots(slots: np.ndarray, seqlens, page: int):
    """The block table the cache writer's slot mapping implies (tokens of each sequence in order)."""
    max_blocks = max(1, max((int(s) + page - 1) // page for s in seqlens))
    bt = np.zeros((len(seqlens), max_blocks), dtype=np.int32)
    t = 0
    for i, s in enumerate(seqlens):
        for lp in range((int(s) + page - 1) // page):
            bt[i, lp] = slots[t + lp * page] // page
        t += int(s)
    return bt


def test_write_then_decode_round_trip():
    """K and V rows written by fp8_paged_cache_write (per-row amax / 448 scales), then decoded with
    those scales: the decode matches the oracle on exactly the bytes and scales that were written."""
    seqlens = [517, 33, 2048, 160]
    h_kv, hd, page = 4, 128, 16
    wi = syn.cache_write_inputs(43, seqlens, h_kv=h_kv, hd=hd, page=page, base_tokens=1024, spare_blocks=4,
                                exp_range=3)
    xk = syn.materialise(wi)
    xv = xk.roll(1, dims=0)  # other rows for V, same layout
    n = wi.num_blocks
    caches, scales = [], []
    for x in (xk, xv):
        c = torch.zeros((n, h_kv, page, hd), dtype=torch.uint8, device=DEV)
        s = torch.ones((n, h_kv, page), dtype=torch.float32, device=DEV)
        fm.paged_cache_write(x.to(DEV), wi.slot_mapping.to(DEV), c, token_scales=s)
        caches.append(c)
        scales.append(s)
    torch.cuda.synchronize()
    assert fm.last_device_error() == 0
    bt = torch.from_numpy(_block_table_from_slots(wi.slot_mapping.numpy(), seqlens, page))
    sl = torch.tensor(seqlens, dtype=torch.int32)
    h_q = 4 * h_kv
    q = syn.gqa_block_q(43, len(seqlens), 1, h_q, hd)
    softmax_scale = hd ** -0.5
    out, lse = fm.paged_gqa_decode_ext(q.to(DEV), caches[0], caches[1], bt.to(DEV), sl.to(DEV), scales[0],
                                       scales[1], softmax_scale, num_splits=2)
    torch.cuda.synchronize()
    ro, rl = oracle.gqa_decode(q[:, 0], caches[0].cpu(), caches[1].cpu(), bt, sl, scales[0].cpu().numpy(),
                               scales[1].cpu().numpy(), softmax_scale)
    assert_close(compare(out[:, 0], lse[:, 0], ro, rl, "bf16"), "bf16")
    assert fm.last_device_error() == 0


XQA = [  # (q_len, group, mask, window, sinks, splits, per_row)
    (3, 4, "causal", 0, False, 1, False),
    (3, 4, "causal", 0, False, 3, False),
    (4, 4, "random", 0, False, 1, False),
    (2, 8, "random", 37, False, 2, False),
    (3, 4, "causal", 1, True, 1, False),
    (1, 8, "causal", 100, True, 4, False),
    (4, 4, "random", 300, True, 3, True),
    (2, 2, "random", 0, True, 1, True),
]


@pytest.mark.parametrize("case", XQA, ids=[f"q{c[0]}_g{c[1]}_{c[2]}_w{c[3]}_s{int(c[4])}_sp{c[5]}_r{int(c[6])}"
                                           for c in XQA])
def test_xqa_options(case):
    q_len, group, mask_kind, window, with_sinks, splits, per_row = case
    h_kv = 2
    h_q = h_kv * group
    seqlens = [700, 3, 2, 0, 129, 1500]  # includes s_k < q_len and an empty cache
    inp = syn.gqa_inputs(44, len(seqlens), seqlens, h_q=h_q, h_kv=h_kv, spare_blocks=5)
    d = _dev_inputs(inp)
    q = syn.gqa_block_q(44, len(seqlens), q_len, h_q)
    mask = syn.spec_mask(44, len(seqlens), q_len) if mask_kind == "random" else None
    sinks = syn.sink_logits(44, h_q) if with_sinks else None
    if per_row:
        shape = tuple(inp.k_cache.shape[:3])
        ks_h = syn.per_row_scales(44, 52, shape, inp.k_scale)
        vs_h = syn.per_row_scales(44, 53, shape, inp.v_scale)
        ks, vs = ks_h.to(DEV), vs_h.to(DEV)
        ks_ref, vs_ref = ks_h.numpy(), vs_h.numpy()
    else:
        ks = torch.tensor([inp.k_scale], dtype=torch.float32, device=DEV)
        vs = torch.tensor([inp.v_scale], dtype=torch.float32, device=DEV)
        ks_ref, vs_ref = inp.k_scale, inp.v_scale
    out, lse = fm.paged_gqa_decode_ext(q.to(DEV), d["kc"], d["vc"], d["bt"], d["sl"], ks, vs, inp.softmax_scale,
                                       spec_mask=None if mask is None else mask.to(DEV), window=window,
                                       sinks=None if sinks is None else sinks.to(DEV), num_splits=splits)
    torch.cuda.synchronize()
    ro, rl = gqa_decode_ext(q, inp.k_cache, inp.v_cache, inp.block_table, inp.seqlens, ks_ref, vs_ref,
                                   inp.softmax_scale, spec_mask=None if mask is None else mask.numpy(),
                                   window=window, sinks=None if sinks is None else sinks.numpy())
    # rows that see no key: out exactly 0 and lse = the sink (or -inf)
    o = out.float().cpu().numpy()
    none = ~np.isfinite(rl) | (np.abs(ro).sum(axis=-1) == 0)
    assert np.all(o[none] == 0)
    l_gpu = lse.cpu().numpy()
    assert np.array_equal(np.isneginf(l_gpu), np.isneginf(rl))
    assert_close(compare(out, lse, ro, rl, "bf16"), "bf16")
    assert fm.last_device_error() == 0


def test_window_on_a_full_grid_runs_unsplit():
    """With a window, a grid that fills the GPU (16 sequences x 8 KV heads) is not split: the
    library's choice is 1, and the unsplit call matches the oracle and a forced 4-way split."""
    h_kv, group, q_len, window = 8, 4, 4, 256
    seqlens = [int(x) for x in np.random.default_rng(45).integers(200, 1400, 16)]
    inp = syn.gqa_inputs(45, len(seqlens), seqlens, h_q=h_kv * group, h_kv=h_kv, spare_blocks=4)
    assert fm.gqa_ext_num_splits(len(seqlens), h_kv, inp.block_table.shape[1] * 16, q_len, window) == 1
    d = _dev_inputs(inp)
    q = syn.gqa_block_q(45, len(seqlens), q_len, h_kv * group)
    mask = syn.spec_mask(45, len(seqlens), q_len)
    sinks = syn.sink_logits(45, h_kv * group)
    ks = torch.tensor([inp.k_scale], dtype=torch.float32, device=DEV)
    vs = torch.tensor([inp.v_scale], dtype=torch.float32, device=DEV)
    runs = {}
    for splits in (0, 4):
        runs[splits] = fm.paged_gqa_decode_ext(q.to(DEV), d["kc"], d["vc"], d["bt"], d["sl"], ks, vs,
                                               inp.softmax_scale, spec_mask=mask.to(DEV), window=window,
                                               sinks=sinks.to(DEV), num_splits=splits)
    torch.cuda.synchronize()
    ro, rl = gqa_decode_ext(q, inp.k_cache, inp.v_cache, inp.block_table, inp.seqlens, inp.k_scale, inp.v_scale,
                            inp.softmax_scale, spec_mask=mask.numpy(), window=window, sinks=sinks.numpy())
    for splits, (out, lse) in runs.items():
        assert_close(compare(out, lse, ro, rl, "bf16"), "bf16")
    assert fm.last_device_error() == 0
