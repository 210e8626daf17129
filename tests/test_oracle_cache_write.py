"""Pins of the cache-write oracle (quantise on write) against facts that do
not come from it.

* E4M3 encoding: torch's own float8_e4m3fn cast (round to nearest even) on
  every value, midpoint and midpoint +- 1 ulp in [-448, 448] and on random
  values; saturation past 448; encode(decode(c)) = c for all 254 finite codes.
* Worked rows derived by hand (``golden/cache_write_rows.txt``): the scale
  amax / 448 of the InfiniCore page's paged_caching bullet, an all-zero row,
  ties in both directions, and a tiny row that takes the 2^64 lift.
* Properties on random rows: the largest element of each row encodes to
  +-448 exactly; every code is within half an E4M3 step of x / scale; slots
  are honoured and nothing else is written.
"""

import os

import numpy as np
import pytest
import torch

from oracle.attention import E4M3_TABLE, e4m3_decode
from oracle.cache_write import e4m3_encode, paged_cache_write, quantise_rows, row_inverse, row_scale
from paged_decode_attention_fp8_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_e4m3(y):
    return torch.from_numpy(np.asarray(y, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_encoder_matches_torch_on_midpoints():
    mags = E4M3_TABLE[:0x7F]
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    ys = np.concatenate([mags.astype(np.float32), mids, np.nextafter(mids, np.float32(0)),
                         np.nextafter(mids, np.float32(1e9))])
    ys = np.concatenate([ys, -ys])
    ys = ys[np.abs(ys) <= 448]
    assert np.array_equal(e4m3_encode(ys), _torch_e4m3(ys))


def test_encoder_matches_torch_on_random_values():
    u = syn.uniform(41, 0, 400000)
    n = syn.normal(41, 1, (400000,))
    y = (n * np.exp2(u * 20.0 - 14.0)).astype(np.float32)            # magnitudes 2^-14 .. 2^6 and more
    y = y[np.abs(y) <= 448]
    assert y.size > 300000
    assert np.array_equal(e4m3_encode(y), _torch_e4m3(y))


def test_encoder_saturates_and_keeps_signs():
    big = np.array([448.0, 448.5, 463.99, 464.0, 1e6, 3.0e38], dtype=np.float32)
    assert np.all(e4m3_encode(big) == 0x7E)
    assert np.all(e4m3_encode(-big) == 0xFE)
    assert e4m3_encode(np.array([0.0]))[0] == 0x00
    assert e4m3_encode(np.array([-0.0]))[0] == 0x80
    assert e4m3_encode(np.array([-1e-30]))[0] == 0x80                # rounds to -0
    with pytest.raises(ValueError):
        e4m3_encode(np.array([np.nan]))


def test_encoder_inverts_the_table():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(e4m3_encode(e4m3_decode(codes)), codes)


def test_worked_rows():
    with open(os.path.join(GOLDEN, "cache_write_rows.txt")) as f:
        rows = [line.split() for line in f if line.strip() and not line.startswith("#")]
    assert len(rows) == 4
    for r in rows:
        semi = r.index(";")
        scale = np.float32(float(r[1]))
        x = np.array([float(v) for v in r[2:semi]], dtype=np.float64)
        codes = np.array([int(v, 16) for v in r[semi + 1:]], dtype=np.uint8)
        amax = np.float32(np.abs(x).max())
        got_scale = row_scale(amax)
        assert got_scale == scale, r[0]
        lift, inv = row_inverse(amax)
        assert np.array_equal(quantise_rows(x, inv, lift), codes), r[0]
        # the same row through the paged write, one token, one head, slot 5 of 2 x 4
        cache = np.full((2, 1, 4, 8), 0x7F, dtype=np.uint8)
        scales = np.full((2, 1, 4), -1.0, dtype=np.float32)
        out, sc = paged_cache_write(x[None, None, :], np.array([5]), cache, 4, token_scales=scales)
        assert np.array_equal(out[1, 0, 1], codes) and sc[1, 0, 1] == scale
        assert np.count_nonzero(out != 0x7F) <= 8 and np.count_nonzero(sc != -1.0) == 1


def _bf16_rows(seed, shape, spread=True):
    v = syn.normal(seed, 0, shape)
    if spread:  # rows of very different magnitudes
        v = v * np.exp2(syn.uniform(seed, 1, shape[0] * shape[1]) * 24.0 - 12.0).reshape(shape[0], shape[1], 1)
    return syn.to_bf16(v).float().numpy().astype(np.float64)


def test_row_max_encodes_to_448_and_codes_are_nearest():
    x = _bf16_rows(42, (64, 4, 128))
    n_blocks, page = 8, 16
    slots = syn.permutation(42, 2, n_blocks * page)[:64]
    cache = np.zeros((n_blocks, 4, page, 128), dtype=np.uint8)
    out, sc = paged_cache_write(x, slots, cache, page, token_scales=np.zeros((n_blocks, 4, page), np.float32))
    for t in range(64):
        blk, off = divmod(int(slots[t]), page)
        for h in range(4):
            row = x[t, h]
            codes = out[blk, h, off]
            s = float(sc[blk, h, off])
            assert s == np.float32(np.float32(np.abs(row).max()) / np.float32(448))
            j = int(np.argmax(np.abs(row)))
            assert codes[j] == (0xFE if row[j] < 0 else 0x7E)
            # nearest: |decode - y| <= half the gap to the neighbouring E4M3 value
            lift, inv = row_inverse(np.float32(np.abs(row).max()))
            y = ((row.astype(np.float32) * lift) * inv).astype(np.float64)
            # y is x / s up to two float32 roundings
            assert np.allclose(y, row / s, rtol=2.0 ** -22, atol=0)
            dec = e4m3_decode(codes)
            mags = E4M3_TABLE[:0x7F]
            k = np.searchsorted(mags, np.abs(dec))
            gap = np.where(k < 0x7E, mags[np.minimum(k + 1, 0x7E)] - mags[k], 32.0)
            gap_below = np.where(k > 0, mags[k] - mags[np.maximum(k - 1, 0)], mags[1])
            assert np.all(np.abs(dec - y) <= np.maximum(gap, gap_below) / 2 + 1e-30)


def test_slots_are_honoured_and_nothing_else_is_written():
    x = _bf16_rows(43, (40, 2, 64), spread=False)
    n_blocks, page = 6, 8
    slots = syn.permutation(43, 3, n_blocks * page)[:40].astype(np.int64)
    slots[::7] = -1
    cache = np.full((n_blocks, 2, page, 64), 0x7F, dtype=np.uint8)
    out, _ = paged_cache_write(x, slots, cache, page, tensor_scale=0.01)
    written = np.zeros((n_blocks, 2, page), dtype=bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        blk, off = divmod(int(s), page)
        written[blk, :, off] = True
        y = x[t].astype(np.float32) * (np.float32(1.0) / np.float32(0.01))   # float32, as defined
        assert np.array_equal(out[blk, :, off], _torch_e4m3(np.clip(y, -448, 448)))
    assert np.all(out[~written] == 0x7F)


def test_all_zero_row_scale_is_one():
    x = np.zeros((1, 1, 16))
    out, sc = paged_cache_write(x, np.array([0]), np.full((1, 1, 1, 16), 0x7F, np.uint8), 1,
                                token_scales=np.zeros((1, 1, 1), np.float32))
    assert sc[0, 0, 0] == 1.0 and np.all(out == 0)
