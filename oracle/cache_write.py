"""CPU oracle for the FP8 (E4M3) paged KV-cache write (quantise on write).

TEST INFRASTRUCTURE ONLY, under the same rule as ``oracle.attention``: only
the test suite, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
may use it, and it shares no code with the CUDA library.

What it computes (InfiniCore "add FP8 blockwise dequantize/GEMM operators and
FP8(E4M3) KV cache support in paged attention", Summary, paged_caching):
every (token, kv_head) row x of head_dim values is stored in the slot the
slot mapping names, as E4M3 codes of x / scale.  Per-row mode: scale =
amax(|x|) / 448, or 1 when the row is all zeros, and the scale is kept in a
[num_blocks, h_kv, page] array; per-tensor mode: one given scale.

The code is an integer decided by floating point, so the oracle takes that
decision in the precision the kernel uses, float32 with round-to-nearest-even
operations: the kept scale is fp32(amax / 448), the codes use its reciprocal
inv = fp32(448 / amax) (one division per row), y = fp32(x * inv), and y is
rounded to the nearest E4M3 value, ties to the even code, saturating at
+-448 (``e4m3_encode``, written from the E4M3 definition: the 256-pattern
table of ``oracle.attention``).  A row with amax < 2^-64 is first multiplied
by 2^64 (exact) so that inv cannot overflow.  Per-tensor mode: inv =
fp32(1 / scale).  Readings where the page is silent: the page gives the
scale and "encode", not the rounding steps, and a multiplication by the
row's reciprocal is taken; a negative slot skips the token (the padding
convention of paged caches); inputs are finite.
"""

from __future__ import annotations

import numpy as np

from .attention import E4M3_TABLE, as_bytes, as_float64, as_int64

E4M3_MAX = 448.0
# magnitudes of codes 0x00 .. 0x7E, increasing (0x7F is NaN)
_MAGNITUDES = E4M3_TABLE[:0x7F]


def e4m3_encode(y) -> np.ndarray:
    """E4M3 codes of the values y: nearest representable value, ties to the
    even code (mantissa bit 0 clear), magnitudes >= 448 saturate to 448, the
    sign is kept (a negative value that rounds to zero gives 0x80).

    The distances below are exact in float64 for float32 inputs: an E4M3
    value's last bit is >= 2^-9 and its first <= 2^8, and for |y| >= 2^-10 the
    float32 y spans at most 2^8 .. 2^-33; below 2^-10 the nearer neighbour is
    0 whatever the rounding of 2^-9 - |y|."""
    y = np.asarray(y, dtype=np.float64)
    if not np.all(np.isfinite(y)):
        raise ValueError("e4m3_encode: non-finite input")
    a = np.abs(y)
    lo = np.searchsorted(_MAGNITUDES, a, side="right") - 1       # _MAGNITUDES[lo] <= a
    lo = np.clip(lo, 0, 0x7E)
    hi = np.minimum(lo + 1, 0x7E)
    d_lo = a - _MAGNITUDES[lo]
    d_hi = _MAGNITUDES[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0) & (hi != lo))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= E4M3_MAX, 0x7E, code)
    sign = np.signbit(y).astype(np.int64) << 7
    return (code | sign).astype(np.uint8)


TINY_AMAX = np.float32(2.0 ** -64)
TINY_LIFT = np.float32(2.0 ** 64)


def row_scale(amax_f32) -> np.ndarray:
    """float32 amax / 448 per row, 1 where amax is 0: the scale the cache keeps."""
    amax = np.asarray(amax_f32, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        s = amax / np.float32(E4M3_MAX)
    return np.where(amax > 0, s, np.float32(1.0)).astype(np.float32)


def row_inverse(amax_f32):
    """(lift, inv) per row, float32: lift = 2^64 where amax < 2^-64, else 1;
    inv = 448 / (amax * lift), 1 where amax is 0."""
    amax = np.asarray(amax_f32, dtype=np.float32)
    lift = np.where(amax < TINY_AMAX, TINY_LIFT, np.float32(1.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = np.float32(E4M3_MAX) / (amax * lift)
    return lift, np.where(amax > 0, inv, np.float32(1.0)).astype(np.float32)


def quantise_rows(x, inv, lift=np.float32(1.0)) -> np.ndarray:
    """E4M3 codes of fp32(fp32(x * lift) * inv); x [..., head_dim], lift and inv broadcast per row."""
    xf = np.asarray(as_float64(x), dtype=np.float32)             # bf16 -> float32 is exact
    y = (xf * np.asarray(lift, dtype=np.float32)) * np.asarray(inv, dtype=np.float32)
    return e4m3_encode(y.astype(np.float32))


def paged_cache_write(x, slot_mapping, cache, page_size: int, tensor_scale=None, token_scales=None):
    """The cache (and per-row scales) after writing x.

    x [n_tokens, h_kv, head_dim] (bf16 values), slot_mapping [n_tokens],
    cache E4M3 bytes [num_blocks, h_kv, page_size, head_dim] (the starting
    contents), token_scales float32 [num_blocks, h_kv, page_size] (starting
    contents) for per-row mode, or tensor_scale (a float) for per-tensor mode.
    Returns (cache bytes, scales or None) as new arrays; rows with a negative
    slot, or a slot past the cache, are not written."""
    if (tensor_scale is None) == (token_scales is None):
        raise ValueError("give exactly one of tensor_scale and token_scales")
    xs = as_float64(x)
    slots = as_int64(slot_mapping)
    out = as_bytes(cache).copy()
    num_blocks, h_kv, page, hd = out.shape
    assert page == page_size and xs.shape[1:] == (h_kv, hd)
    scales = None if token_scales is None else np.asarray(as_float64(token_scales), dtype=np.float32).copy()
    for t in range(xs.shape[0]):
        s = int(slots[t])
        if s < 0 or s >= num_blocks * page:
            continue
        blk, off = divmod(s, page)
        rows = xs[t]                                              # [h_kv, hd]
        if scales is not None:
            amax = np.abs(rows).max(axis=1).astype(np.float32)
            scales[blk, :, off] = row_scale(amax)
            lift, inv = row_inverse(amax)
            out[blk, :, off, :] = quantise_rows(rows, inv[:, None], lift[:, None])
        else:
            out[blk, :, off, :] = quantise_rows(rows, np.float32(1.0) / np.float32(tensor_scale))
    return out, scales
