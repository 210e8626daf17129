"""FP8 paged KV-cache write (quantise on write) on the GPU against the oracle,
through the C ABI.  Codes and per-row scales are integers / exact floats
decided in float32 on both sides, so every comparison is bit-exact.

Shapes follow the InfiniCore paged_caching bullet (per-row scales
[num_blocks, h_kv, page], GQA layout h_kv 8, head_dim 128, page 16) and the
dense MLA cache (one 576-wide row per token, page 64, one per-tensor scale).
"""

import numpy as np
import pytest
import torch

import paged_decode_attention_fp8_gb300 as fm
from oracle.cache_write import paged_cache_write as ref_write
from oracle.cache_write import quantise_rows, row_inverse, row_scale
from paged_decode_attention_fp8_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

POISON = 0x7F
SENTINEL = -3.0


def _run(inp, x, per_row=True, tensor_scale=None, h_kv=None, hd=None):
    dev = torch.device("cuda")
    h_kv = h_kv or x.shape[1]
    hd = hd or x.shape[2]
    cache = torch.full((inp.num_blocks, h_kv, inp.page, hd), POISON, dtype=torch.uint8, device=dev)
    scales = torch.full((inp.num_blocks, h_kv, inp.page), SENTINEL, dtype=torch.float32, device=dev) if per_row \
        else None
    ts = None if per_row else torch.tensor([tensor_scale], dtype=torch.float32, device=dev)
    fm.paged_cache_write(x.to(dev), inp.slot_mapping.to(dev), cache, tensor_scale=ts, token_scales=scales)
    torch.cuda.synchronize()
    return cache.cpu().numpy(), None if scales is None else scales.cpu().numpy()


def _ref(inp, x, per_row=True, tensor_scale=None):
    n = inp.num_blocks
    h_kv, hd = x.shape[1], x.shape[2]
    cache = np.full((n, h_kv, inp.page, hd), POISON, dtype=np.uint8)
    if per_row:
        return ref_write(x, inp.slot_mapping, cache, inp.page,
                         token_scales=np.full((n, h_kv, inp.page), SENTINEL, dtype=np.float32))
    return ref_write(x, inp.slot_mapping, cache, inp.page, tensor_scale=tensor_scale)


# every lane-group shape the kernel has: one to three chunks of 8 values per
# lane at 1 lane, two or three at 2-16 lanes, two to four at 32; 40, 80, 200,
# 328 and 576 leave some lanes of each group without a chunk
@pytest.mark.parametrize("hd", [8, 16, 24, 32, 40, 64, 80, 128, 192, 200, 256, 328, 512, 576, 1024])
def test_per_row_head_dims(hd):
    # ragged lengths (partial last blocks), padding slots, several row groups per warp
    inp = syn.cache_write_inputs(21, [37, 5, 70], h_kv=2, hd=hd, page=16, base_tokens=64, spare_blocks=3,
                                 pad_tokens=4)
    x = syn.materialise(inp)
    got, gs = _run(inp, x)
    want, ws = _ref(inp, x)
    assert np.array_equal(got, want)
    assert np.array_equal(gs.view(np.uint32), ws.view(np.uint32))
    assert fm.last_device_error() == 0


def test_gqa_layout_per_row_and_untouched_slots():
    seqlens = syn.uniform_seqlens(22, 6, 1, 300)
    inp = syn.cache_write_inputs(22, seqlens, h_kv=8, hd=128, page=16, base_tokens=512, spare_blocks=5,
                                 pad_tokens=9)
    x = syn.materialise(inp)
    got, gs = _run(inp, x)
    want, ws = _ref(inp, x)
    assert np.array_equal(got, want)
    assert np.array_equal(gs.view(np.uint32), ws.view(np.uint32))
    # slots nothing maps to keep their bytes and scales
    assert (got == POISON).sum() >= 5 * 8 * 16 * 128
    assert (gs == SENTINEL).sum() >= 5 * 8 * 16


def test_mla_layout_per_tensor_scale():
    # the dense MLA cache: [num_pages, 64, 576], one row per token, one scale
    inp = syn.cache_write_inputs(23, [130, 64, 1, 200], h_kv=1, hd=576, page=64, base_tokens=256, spare_blocks=2)
    x = syn.materialise(inp)
    vals = x.float().numpy()
    scale = float(np.float32(np.abs(vals).max() / 448.0) * np.float32(0.5))   # half: the largest rows saturate
    dev = torch.device("cuda")
    cache = torch.full((inp.num_blocks, 64, 576), POISON, dtype=torch.uint8, device=dev)
    ts = torch.tensor([scale], dtype=torch.float32, device=dev)
    fm.paged_cache_write(x[:, 0, :].to(dev), inp.slot_mapping.to(dev), cache, tensor_scale=ts)
    torch.cuda.synchronize()
    want, _ = _ref(inp, x, per_row=False, tensor_scale=scale)
    assert np.array_equal(cache.cpu().numpy(), want[:, 0])
    assert ((want == 0x7E) | (want == 0xFE)).any()                     # saturation was exercised
    assert fm.last_device_error() == 0


def test_typed_cache_and_strided_rows():
    # a float8_e4m3fn cache, and x as a view with padding between tokens
    inp = syn.cache_write_inputs(24, [50, 33], h_kv=4, hd=64, page=16, base_tokens=83)
    x = syn.materialise(inp)
    dev = torch.device("cuda")
    padded = torch.zeros((x.shape[0], 4 * 64 + 16), dtype=torch.bfloat16, device=dev)
    padded[:, :256] = x.reshape(x.shape[0], 256).to(dev)
    xv = padded[:, :256].view(x.shape[0], 4, 64)
    assert xv.stride(0) == 272
    cache = torch.full((inp.num_blocks, 4, 16, 64), POISON, dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
    scales = torch.full((inp.num_blocks, 4, 16), SENTINEL, dtype=torch.float32, device=dev)
    fm.paged_cache_write(xv, inp.slot_mapping.to(dev), cache, token_scales=scales)
    torch.cuda.synchronize()
    want, ws = _ref(inp, x)
    assert np.array_equal(cache.view(torch.uint8).cpu().numpy(), want)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), ws.view(np.uint32))


def test_zero_rows_and_extreme_magnitudes():
    inp = syn.cache_write_inputs(25, [40], h_kv=2, hd=128, page=16, base_tokens=40, exp_range=0)
    x = syn.materialise(inp).float()
    x[3] = 0.0                                   # an all-zero token: scale 1, codes 0
    x[5, 1] = 0.0                                # one all-zero head
    x[7] *= 2.0 ** 100                           # huge and tiny rows (still bf16 normals)
    x[8] *= 2.0 ** -100
    x[9, 0, :] = 0.0
    x[9, 0, 17] = -2.0 ** -120                   # one tiny nonzero value in a row
    x[10, 1, :] = 0.0
    x[10, 1, 40] = 2.0 ** -130                   # a bf16 subnormal: the row's amax must keep it
    x = x.to(torch.bfloat16)
    got, gs = _run(inp, x)
    want, ws = _ref(inp, x)
    assert np.array_equal(got, want)
    assert np.array_equal(gs.view(np.uint32), ws.view(np.uint32))
    s3 = int(inp.slot_mapping[3])
    assert np.all(gs[s3 // 16, :, s3 % 16] == 1.0)


def test_bad_slot_is_reported_and_skipped():
    inp = syn.cache_write_inputs(26, [20], h_kv=2, hd=64, page=16, base_tokens=20, spare_blocks=1)
    slots = inp.slot_mapping.clone()
    slots[4] = inp.num_blocks * 16               # one past the cache
    inp.slot_mapping = slots
    x = syn.materialise(inp)
    fm.last_device_error()
    got, gs = _run(inp, x)
    assert fm.last_device_error() == fm.DEV_BAD_SLOT
    want, ws = _ref(inp, x)                      # the oracle skips it as well
    assert np.array_equal(got, want)
    assert np.array_equal(gs.view(np.uint32), ws.view(np.uint32))


def test_empty_write_is_a_no_op():
    dev = torch.device("cuda")
    cache = torch.full((2, 1, 16, 64), POISON, dtype=torch.uint8, device=dev)
    fm.paged_cache_write(torch.empty((0, 1, 64), dtype=torch.bfloat16, device=dev),
                         torch.empty((0,), dtype=torch.int32, device=dev), cache,
                         token_scales=torch.zeros((2, 1, 16), dtype=torch.float32, device=dev))
    torch.cuda.synchronize()
    assert bool((cache == POISON).all())


def test_full_size_sampled():
    # the bench workload: K rows of 32 sequences with contexts uniform in [1024, 16384],
    # 8 KV heads x 128, page 16, per-row scales; rows sampled for the oracle
    seqlens = syn.uniform_seqlens(5, 32, 1024, 16384)
    inp = syn.cache_write_inputs(5, seqlens)
    dev = torch.device("cuda")
    x = syn.materialise(inp, device=dev)
    n = x.shape[0]
    cache = torch.full((inp.num_blocks, 8, 16, 128), POISON, dtype=torch.uint8, device=dev)
    scales = torch.full((inp.num_blocks, 8, 16), SENTINEL, dtype=torch.float32, device=dev)
    fm.paged_cache_write(x, inp.slot_mapping.to(dev), cache, token_scales=scales)
    torch.cuda.synchronize()
    assert fm.last_device_error() == 0
    sample = np.unique(np.concatenate([syn.randint(5, 30, 3000, 0, n - 1), [0, n - 1]]))
    rows = syn.materialise(inp, sample).float().numpy().astype(np.float64)   # built on the host
    slots = inp.slot_mapping.numpy()[sample].astype(np.int64)
    blk, off = slots // 16, slots % 16
    got = cache[torch.from_numpy(blk).to(dev), :, torch.from_numpy(off).to(dev)].cpu().numpy()
    gsc = scales[torch.from_numpy(blk).to(dev), :, torch.from_numpy(off).to(dev)].cpu().numpy()
    amax = np.abs(rows).max(axis=2).astype(np.float32)
    want_sc = row_scale(amax)
    lift, inv = row_inverse(amax)
    want = quantise_rows(rows, inv[:, :, None], lift[:, :, None])
    assert np.array_equal(gsc.view(np.uint32), want_sc.view(np.uint32))
    assert np.array_equal(got, want)
    # every slot of the pool that a token maps to was written (no sentinel left)
    assert int((scales == SENTINEL).sum()) == (inp.num_blocks * 16 - n) * 8
