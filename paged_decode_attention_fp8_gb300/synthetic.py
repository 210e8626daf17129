"""Seeded synthetic inputs for FP8 paged decode attention.

This module only draws numbers and lays them out; it computes no part of the
attention.  Both the CUDA path and the fp64 oracle consume what it returns,
byte for byte.

Recipe (shapes follow the workloads on the FlashMLA "update fp8 support" page,
the aiter sparse_mla_fwd page and the InfiniCore paged-attention page):

* random numbers: a counter-based splitmix64 stream per (seed, purpose),
  mapped to (0, 1] and then to N(0, 1) by Box-Muller, all in float64;
* Q: N(0, 1) rounded to bf16;
* KV: N(0, 1) over the valid token slots, one per-tensor scale
  ``amax / 448`` (stored as float32), then E4M3 ("fn" encoding) of
  ``x / scale`` clamped to +-448 -- the cast itself is torch's
  ``float8_e4m3fn`` conversion, a library routine;
* paging: the used pages are placed at a seeded random permutation of the
  physical pool; spare pages and every slot past a sequence's length hold
  the byte 0x7F (an E4M3 NaN), so any read that should not happen shows up.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

E4M3_MAX = 448.0
POISON_BYTE = 0x7F

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix64(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def u64_stream(seed: int, purpose: int, n: int) -> np.ndarray:
    """n splitmix64 outputs for the stream keyed by (seed, purpose)."""
    key = _mix64(np.array([(seed * 1_000_003 + purpose) & 0xFFFFFFFFFFFFFFFF],
                          dtype=np.uint64))[0]
    idx = np.arange(1, n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + idx * _GOLDEN)


def uniform(seed: int, purpose: int, n: int) -> np.ndarray:
    """Uniform float64 in (0, 1]."""
    u = u64_stream(seed, purpose, n) >> np.uint64(11)
    return (u.astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


def normal(seed: int, purpose: int, shape) -> np.ndarray:
    """N(0, 1) float64 by Box-Muller."""
    n = int(np.prod(shape))
    m = (n + 1) // 2
    u1 = uniform(seed, 2 * purpose, m)
    u2 = uniform(seed, 2 * purpose + 1, m)
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.concatenate([r * np.cos(2.0 * math.pi * u2), r * np.sin(2.0 * math.pi * u2)])
    return z[:n].reshape(shape)


def permutation(seed: int, purpose: int, n: int) -> np.ndarray:
    keys = u64_stream(seed, purpose, n)
    return np.argsort(keys, kind="stable").astype(np.int64)


def randint(seed: int, purpose: int, n: int, lo: int, hi: int) -> np.ndarray:
    """Integers uniform in [lo, hi] (inclusive)."""
    span = hi - lo + 1
    u = uniform(seed, purpose, n)
    return np.minimum(lo + np.floor(u * span).astype(np.int64), hi)


def to_bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def per_tensor_scale(values: np.ndarray) -> float:
    """amax / 448 as the float32 value both sides use (1.0 for an all-zero tensor)."""
    amax = float(np.max(np.abs(values))) if values.size else 0.0
    return float(np.float32(amax / E4M3_MAX)) if amax > 0 else 1.0


def to_e4m3_bytes(x: np.ndarray, scale) -> np.ndarray:
    """E4M3 bytes of x / scale (torch's float8_e4m3fn cast after clamping); scale is a float or an
    array that broadcasts against x."""
    y = np.clip(np.asarray(x, dtype=np.float64) / scale, -E4M3_MAX, E4M3_MAX)
    t = torch.from_numpy(np.ascontiguousarray(y, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


# --------------------------------------------------------------------------
# Dense MLA (d = 576 = 512 latent + 64 RoPE, dv = 512, one KV head, page 64)
# --------------------------------------------------------------------------

MLA_D = 576
MLA_DV = 512
MLA_PAGE = 64


@dataclass
class MLAInputs:
    q: torch.Tensor            # bf16 [b, s_q, h_q, 576]
    kv_cache: torch.Tensor     # uint8 (E4M3 bytes) [num_pages, 64, 576]
    block_table: torch.Tensor  # int32 [b, max_pages]
    seqlens: torch.Tensor      # int32 [b]
    kv_scale: float            # float32 value
    softmax_scale: float
    causal: bool

    @property
    def b(self):
        return self.q.shape[0]

    @property
    def s_q(self):
        return self.q.shape[1]

    @property
    def h_q(self):
        return self.q.shape[2]


def _mla_layout(seed: int, seqlens: np.ndarray, spare_pages: int, page_order=None):
    """Page placement shared by the MLA generators: (num_pages, used pages,
    pages per sequence, block table) with the used pages at a seeded random
    permutation of the pool and every unused table entry naming a spare page."""
    b = seqlens.shape[0]
    n_pages = (seqlens + MLA_PAGE - 1) // MLA_PAGE
    used = int(n_pages.sum())
    num_pages = max(used + spare_pages, 1)
    perm = permutation(seed, 1, num_pages) if page_order is None else np.asarray(page_order)
    max_pages = max(int(n_pages.max()) if b else 1, 1)
    fill = int(perm[used]) if num_pages > used else 0
    block_table = np.full((b, max_pages), fill, dtype=np.int32)
    k = 0
    for i in range(b):
        for p in range(int(n_pages[i])):
            block_table[i, p] = perm[k + p]
        k += int(n_pages[i])
    return num_pages, used, n_pages, block_table


def _mla_valid(seqlens: np.ndarray, used: int, n_pages: np.ndarray) -> np.ndarray:
    """[used * 64] mask of the rows that hold a key (the used pages in sequence order)."""
    valid = np.zeros(used * MLA_PAGE, dtype=bool)
    k = 0
    for i in range(seqlens.shape[0]):
        lo = k * MLA_PAGE
        valid[lo: lo + int(seqlens[i])] = True
        k += int(n_pages[i])
    return valid


def _mla_place(enc: np.ndarray, valid: np.ndarray, num_pages: int, used: int, n_pages: np.ndarray,
               block_table: np.ndarray) -> np.ndarray:
    """The cache [num_pages, 64, 576]: the used pages' encoded rows (sequence
    order) at their block-table entries, 0x7F everywhere else."""
    enc = enc.reshape(used * MLA_PAGE, MLA_D)
    enc[~valid] = POISON_BYTE
    enc = enc.reshape(used, MLA_PAGE, MLA_D)
    cache = np.full((num_pages, MLA_PAGE, MLA_D), POISON_BYTE, dtype=np.uint8)
    k = 0
    for i in range(n_pages.shape[0]):
        for p in range(int(n_pages[i])):
            cache[block_table[i, p]] = enc[k + p]
        k += int(n_pages[i])
    return cache


def _mla_cache(vals: np.ndarray, seqlens: np.ndarray, num_pages: int, used: int, n_pages: np.ndarray,
               block_table: np.ndarray, scale: float | None = None):
    """E4M3 cache [num_pages, 64, 576] holding ``vals`` (the used pages'
    rows in sequence order), every slot past a sequence end and every spare
    page poisoned with 0x7F; the scale is amax / 448 over the valid rows
    unless given."""
    valid = _mla_valid(seqlens, used, n_pages)
    if scale is None:
        scale = per_tensor_scale(vals[valid])
    cache = _mla_place(to_e4m3_bytes(vals, scale), valid, num_pages, used, n_pages, block_table)
    return cache, scale


def mla_inputs(seed: int, b: int, s_q: int, h_q: int, seqlens, causal: bool = True,
               spare_pages: int = 0, softmax_scale: float | None = None,
               page_order: np.ndarray | None = None, value_pages: int | None = None) -> MLAInputs:
    """Paged MLA decode inputs.  ``seqlens`` is a list of cache lengths.

    Every cached value is an N(0, 1) draw.  By default each used page gets
    its own draws; with ``value_pages`` = n (large batches, e.g. 128 x 8196
    tokens) n distinct pages of draws are made and every used page copies
    one of them, chosen by a seeded index, so the generator's time and host
    memory stay bounded (the kernels see ordinary pages; which pages share
    values does not matter to them, and the oracle reads the same bytes)."""
    seqlens = np.asarray(seqlens, dtype=np.int64)
    assert seqlens.shape == (b,)
    num_pages, used, n_pages, block_table = _mla_layout(seed, seqlens, spare_pages, page_order)
    if value_pages is None:
        vals = normal(seed, 2, (max(used, 1) * MLA_PAGE, MLA_D))[: used * MLA_PAGE]
        cache, scale = _mla_cache(vals, seqlens, num_pages, used, n_pages, block_table)
    else:
        # amax / 448 over the valid rows from the pool's per-row maxima; the
        # pool is encoded once and its pages copied
        pool = normal(seed, 2, (value_pages, MLA_PAGE, MLA_D))
        pick = randint(seed, 4, max(used, 1), 0, value_pages - 1)[:used]
        valid = _mla_valid(seqlens, used, n_pages)
        row_amax = np.abs(pool).max(axis=2)[pick].reshape(-1)
        amax = float(row_amax[valid].max()) if valid.any() else 0.0
        scale = float(np.float32(amax / E4M3_MAX)) if amax > 0 else 1.0
        cache = _mla_place(to_e4m3_bytes(pool, scale)[pick], valid, num_pages, used, n_pages, block_table)
    q = to_bf16(normal(seed, 3, (b, s_q, h_q, MLA_D)))
    if softmax_scale is None:
        softmax_scale = float(np.float32(1.0 / math.sqrt(MLA_D)))
    return MLAInputs(q=q, kv_cache=torch.from_numpy(cache),
                     block_table=torch.from_numpy(block_table),
                     seqlens=torch.from_numpy(seqlens.astype(np.int32)),
                     kv_scale=scale, softmax_scale=softmax_scale, causal=causal)


def mla_row_scaled_inputs(seed: int, b: int, s_q: int, h_q: int, seqlens, causal: bool = True,
                          spare_pages: int = 0, value_pages: int | None = None, spread: float = 3.0):
    """Dense MLA inputs with one scale per cached row: (inputs, scales float32 [num_pages, 1, 64]).

    Row j holds N(0, 1) draws x_j stored as E4M3(x_j / sigma_j) with sigma_j = (amax_j / 448) 2^v_j,
    v_j uniform in [0, spread]: the keys keep the statistics of ``mla_inputs`` while the scales span
    a factor 2^spread and the codes use less of the E4M3 range as v_j grows.  ``inputs.kv_scale`` is
    1.0 and unused.  With ``value_pages`` = n, n pages of draws and their row scales are made and each
    used page copies one of them (codes and scales), as in ``mla_inputs``.  Spare pages and rows past
    a sequence end hold 0x7F with scale 1."""
    seqlens = np.asarray(seqlens, dtype=np.int64)
    assert seqlens.shape == (b,)
    num_pages, used, n_pages, block_table = _mla_layout(seed, seqlens, spare_pages)
    n_pool = max(used, 1) if value_pages is None else value_pages
    pool = normal(seed, 2, (n_pool, MLA_PAGE, MLA_D))
    amax = np.abs(pool).max(axis=2)
    v = uniform(seed, 5, n_pool * MLA_PAGE).reshape(n_pool, MLA_PAGE) * spread
    sigma = (amax / E4M3_MAX * np.exp2(v)).astype(np.float32)
    codes = to_e4m3_bytes(pool, sigma.astype(np.float64)[:, :, None])
    pick = np.arange(used) if value_pages is None else randint(seed, 4, max(used, 1), 0, value_pages - 1)[:used]
    valid = _mla_valid(seqlens, used, n_pages)
    cache = _mla_place(codes[pick], valid, num_pages, used, n_pages, block_table)
    rows = np.ones((num_pages, MLA_PAGE), dtype=np.float32)
    k = 0
    for i in range(b):
        for p in range(int(n_pages[i])):
            rows[block_table[i, p]] = sigma[pick[k + p]]
        k += int(n_pages[i])
    q = to_bf16(normal(seed, 3, (b, s_q, h_q, MLA_D)))
    inp = MLAInputs(q=q, kv_cache=torch.from_numpy(cache), block_table=torch.from_numpy(block_table),
                    seqlens=torch.from_numpy(seqlens.astype(np.int32)), kv_scale=1.0,
                    softmax_scale=float(np.float32(1.0 / math.sqrt(MLA_D))), causal=causal)
    return inp, torch.from_numpy(rows.reshape(num_pages, 1, MLA_PAGE))


def mla_peaky_inputs(seed: int, b: int = 2, h_q: int = 64, s_k: int = 2048,
                     spare_pages: int = 4) -> MLAInputs:
    """Dense MLA inputs in which one key per sequence scores +9 above the
    others (s_q = 1, no causal mask): the sparse peaky construction carried
    over to the 576-wide rows.

    Latent dims [0, 256) carry the score and [256, 512) the values; Q is 0 on
    dims [256, 576) (so the RoPE keys, N(0, 1), add nothing).  Tail keys are 0
    on [0, 256) and w + 0.1 N(0, 1) on [256, 512); the peak key (at a seeded
    position) holds kappa on dim 0, 0 on [1, 256) and z on [256, 512).
    kappa is the cache's largest magnitude, so it encodes to exactly 448 and
    the peak scores softmax_scale * 7 * 448 * kv_scale = 9 up to float32
    rounding of the scales, every tail key exactly 0.  With s_k = 2048 the
    2047 tail keys carry e^-9 * 2047 / (1 + e^-9 * 2047) = 0.2017 of the
    weight, so the output on [256, 512) is about 0.8 z + 0.2 w."""
    seqlens = np.full(b, s_k, dtype=np.int64)
    num_pages, used, n_pages, block_table = _mla_layout(seed, seqlens, spare_pages)
    softmax_scale = float(np.float32(1.0 / math.sqrt(MLA_D)))
    kappa = PEAKY_MARGIN / (softmax_scale * PEAKY_Q0)
    kv_scale = float(np.float32(kappa / E4M3_MAX))
    half = SPARSE_D // 2
    w = normal(seed, 11, (half,))
    z = normal(seed, 12, (half,))
    vals = np.zeros((used * MLA_PAGE, MLA_D))
    vals[:, 512:] = normal(seed, 15, (used * MLA_PAGE, MLA_D - 512))
    peaks = randint(seed, 14, b, 0, s_k - 1)
    k = 0
    for i in range(b):
        lo = k * MLA_PAGE
        vals[lo:lo + s_k, half:512] = w[None, :] + 0.1 * normal(seed, 20 + i, (s_k, half))
        j = lo + int(peaks[i])
        vals[j, :512] = 0.0
        vals[j, 0] = E4M3_MAX * kv_scale
        vals[j, half:512] = z
        k += int(n_pages[i])
    cache, _ = _mla_cache(vals, seqlens, num_pages, used, n_pages, block_table, scale=kv_scale)
    q = np.zeros((b, 1, h_q, MLA_D))
    q[..., 0] = PEAKY_Q0
    q[..., 1:half] = normal(seed, 30, (b, 1, h_q, half - 1))
    return MLAInputs(q=to_bf16(q), kv_cache=torch.from_numpy(cache),
                     block_table=torch.from_numpy(block_table),
                     seqlens=torch.from_numpy(seqlens.astype(np.int32)),
                     kv_scale=kv_scale, softmax_scale=softmax_scale, causal=False)


def uniform_seqlens(seed: int, b: int, lo: int, hi: int) -> list[int]:
    return [int(x) for x in randint(seed, 7, b, lo, hi)]


# --------------------------------------------------------------------------
# Sparse top-k MLA (rope-free d = dv = 512, one flat cache of rows)
# --------------------------------------------------------------------------

SPARSE_D = 512


@dataclass
class SparseInputs:
    q: torch.Tensor          # bf16 [s_q, h_q, 512]
    kv_cache: torch.Tensor   # uint8 [num_tokens, 512]
    topk_idx: torch.Tensor   # int32 [s_q, topk]; -1 = skip
    kv_scale: float
    softmax_scale: float


def sparse_inputs(seed: int, s_q: int, h_q: int = 16, num_tokens: int = 131072,
                  topk: int = 2048, index_rule: str = "permutation") -> SparseInputs:
    """Top-k sparse MLA inputs: each query token's topk distinct cache rows.

    index_rule "permutation": token t takes the first topk entries of its own
    seeded permutation of the rows.  "affine" (large batches, num_tokens a
    power of two): one seeded permutation P of the rows, and token t takes
    P[(a_t k + b_t) mod num_tokens] for k < topk with a_t odd -- distinct,
    since multiplying by an odd number permutes the residues -- drawn for all
    tokens at once."""
    vals = normal(seed, 2, (num_tokens, SPARSE_D))
    scale = per_tensor_scale(vals)
    cache = to_e4m3_bytes(vals, scale)
    if index_rule == "permutation":
        idx = np.empty((s_q, topk), dtype=np.int32)
        for t in range(s_q):
            idx[t] = permutation(seed, 100 + t, num_tokens)[:topk]
    elif index_rule == "affine":
        if num_tokens & (num_tokens - 1) or topk > num_tokens:
            raise ValueError("the affine index rule needs a power-of-two cache of at least topk rows")
        perm = permutation(seed, 99, num_tokens).astype(np.int64)
        a = randint(seed, 97, s_q, 0, num_tokens // 2 - 1) * 2 + 1
        b = randint(seed, 98, s_q, 0, num_tokens - 1)
        k = np.arange(topk, dtype=np.int64)
        idx = perm[(a[:, None] * k[None, :] + b[:, None]) & (num_tokens - 1)].astype(np.int32)
    else:
        raise ValueError(f"index rule {index_rule!r}")
    q = to_bf16(normal(seed, 3, (s_q, h_q, SPARSE_D)))
    return SparseInputs(q=q, kv_cache=torch.from_numpy(cache), topk_idx=torch.from_numpy(idx),
                        kv_scale=scale,
                        softmax_scale=float(np.float32(1.0 / math.sqrt(SPARSE_D))))


PEAKY_Q0 = 7.0          # 1.75 * 2**2: exact in bf16 and, after a power-of-two row scale, in E4M3
PEAKY_MARGIN = 9.0      # key 0 scores this much above every other key


def sparse_peaky_inputs(seed: int, s_q: int = 2, h_q: int = 16, num_tokens: int = 131072,
                        topk: int = 2048) -> SparseInputs:
    """One key per query token scores +9 above 2047 keys that score exactly 0.

    Dims [0, 256) carry the score, dims [256, 512) carry the values: Q is 0
    there, the tail keys hold w + 0.1 N(0, 1) and key 0 holds z, so the output
    on those dims is about 0.8 z + 0.2 w.  Key 0's dim 0 is the cache's
    largest magnitude, so it encodes to exactly 448 and its score is
    softmax_scale * 7 * 448 * kv_scale = 9 up to float32 rounding of the scales.
    """
    softmax_scale = float(np.float32(1.0 / math.sqrt(SPARSE_D)))
    kappa = PEAKY_MARGIN / (softmax_scale * PEAKY_Q0)     # true value of key 0's dim 0
    kv_scale = float(np.float32(kappa / E4M3_MAX))
    half = SPARSE_D // 2
    w = normal(seed, 11, (half,))
    z = normal(seed, 12, (half,))
    vals = np.zeros((num_tokens, SPARSE_D))
    idx = np.empty((s_q, topk), dtype=np.int32)
    perm = permutation(seed, 13, num_tokens)
    for t in range(s_q):
        rows = perm[t * topk:(t + 1) * topk]
        key0 = rows[int(randint(seed, 14 + t, 1, 0, topk - 1)[0])]
        vals[rows, half:] = w[None, :] + 0.1 * normal(seed, 20 + t, (topk, half))
        vals[key0, :] = 0.0
        vals[key0, 0] = E4M3_MAX * kv_scale
        vals[key0, half:] = z
        idx[t] = rows
    cache = to_e4m3_bytes(vals, kv_scale)
    q = np.zeros((s_q, h_q, SPARSE_D))
    q[:, :, 0] = PEAKY_Q0
    q[:, :, 1:half] = normal(seed, 30, (s_q, h_q, half - 1))
    return SparseInputs(q=to_bf16(q), kv_cache=torch.from_numpy(cache),
                        topk_idx=torch.from_numpy(idx), kv_scale=kv_scale,
                        softmax_scale=softmax_scale)


# --------------------------------------------------------------------------
# GQA paged decode (separate K / V caches [num_blocks, h_kv, page, head_dim])
# --------------------------------------------------------------------------


@dataclass
class GQAInputs:
    q: torch.Tensor           # bf16 [bs, h_q, hd]
    k_cache: torch.Tensor     # uint8 [num_blocks, h_kv, page, hd]
    v_cache: torch.Tensor     # uint8 [num_blocks, h_kv, page, hd]
    block_table: torch.Tensor # int32 [bs, max_blocks]
    seqlens: torch.Tensor     # int32 [bs]
    k_scale: float
    v_scale: float
    softmax_scale: float


def gqa_inputs(seed: int, bs: int, seqlens, h_q: int = 32, h_kv: int = 8, hd: int = 128,
               page: int = 16, spare_blocks: int = 0, value_blocks: int | None = None) -> GQAInputs:
    """Paged GQA decode inputs: separate E4M3 K and V caches [num_blocks,
    h_kv, page, hd], each with its per-tensor scale amax / 448 over the
    valid rows; the used blocks sit at a seeded random permutation of the
    pool, spare blocks and slots past a sequence end hold 0x7F.  With
    ``value_blocks`` = n, n distinct blocks of N(0, 1) draws are made per
    cache and every used block copies one of them (seeded choice), which
    bounds the generator's time and memory for large batches."""
    seqlens = np.asarray(seqlens, dtype=np.int64)
    n_blocks = (seqlens + page - 1) // page
    used = int(n_blocks.sum())
    num_blocks = max(used + spare_blocks, 1)
    perm = permutation(seed, 1, num_blocks)
    max_blocks = max(int(n_blocks.max()) if bs else 1, 1)
    fill = int(perm[used]) if num_blocks > used else 0
    block_table = np.full((bs, max_blocks), fill, dtype=np.int32)
    # used block u belongs to sequence seq[u] as its logical block lp[u]
    seq = np.repeat(np.arange(bs), n_blocks)
    first = np.concatenate([[0], np.cumsum(n_blocks)[:-1]]).astype(np.int64) if bs else np.zeros(0, np.int64)
    lp = np.arange(used) - np.repeat(first, n_blocks)
    block_table[seq, lp] = perm[:used]
    rows_valid = np.minimum(page, seqlens[seq] - lp * page) if used else np.zeros(0, np.int64)
    valid = np.arange(page)[None, :] < rows_valid[:, None]
    caches, scales = [], []
    for purpose in (2, 4):
        if value_blocks is None:
            vals = normal(seed, purpose, (max(used, 1), h_kv, page, hd))[:used]
            vmask = np.broadcast_to(valid[:, None, :, None], vals.shape)
            scale = per_tensor_scale(vals[vmask])
            enc = to_e4m3_bytes(vals, scale)
        else:
            # the same amax / 448 over the valid rows, taken from per-row maxima
            # of the pool; the pool is encoded once and its blocks copied
            pool = normal(seed, purpose, (value_blocks, h_kv, page, hd))
            pick = randint(seed, purpose + 10, max(used, 1), 0, value_blocks - 1)[:used]
            row_amax = np.abs(pool).max(axis=3)[pick]  # [used, h_kv, page]
            amax = float(row_amax[np.broadcast_to(valid[:, None, :], row_amax.shape)].max()) if used else 0.0
            scale = float(np.float32(amax / E4M3_MAX)) if amax > 0 else 1.0
            enc = to_e4m3_bytes(pool, scale)[pick]
            vmask = np.broadcast_to(valid[:, None, :, None], enc.shape)
        enc[~vmask] = POISON_BYTE
        cache = np.full((num_blocks, h_kv, page, hd), POISON_BYTE, dtype=np.uint8)
        cache[perm[:used]] = enc
        caches.append(torch.from_numpy(cache))
        scales.append(scale)
    q = to_bf16(normal(seed, 3, (bs, h_q, hd)))
    return GQAInputs(q=q, k_cache=caches[0], v_cache=caches[1],
                     block_table=torch.from_numpy(block_table),
                     seqlens=torch.from_numpy(seqlens.astype(np.int32)),
                     k_scale=scales[0], v_scale=scales[1],
                     softmax_scale=float(np.float32(1.0 / math.sqrt(hd))))


# ------------------------------------------------------ cache write inputs --


@dataclass
class CacheWriteInputs:
    base: torch.Tensor         # bf16 [base_tokens, h_kv, hd]: N(0, 1) rows
    exponent: np.ndarray       # int64 [n_tokens]: token t is base[t % base_tokens] * 2^exponent[t]
    slot_mapping: torch.Tensor # int32 [n_tokens]: block * page + offset, -1 = padding
    num_blocks: int
    page: int
    seqlens: np.ndarray        # int64 [bs]: tokens of each sequence, in token order


def cache_write_inputs(seed: int, seqlens, h_kv: int = 8, hd: int = 128, page: int = 16,
                       base_tokens: int = 4096, spare_blocks: int = 0, pad_tokens: int = 0,
                       exp_range: int = 8) -> CacheWriteInputs:
    """New K (or V) rows of whole sequences and the slots a paged cache gives them.

    Sequence i's tokens take the blocks of a seeded random permutation of the
    pool in order (as in ``gqa_inputs``); ``pad_tokens`` slots of -1 are mixed
    in at seeded positions.  Row values: a block of ``base_tokens`` N(0, 1)
    rows (bf16) repeated, token t scaled by 2^e (e uniform in
    [-exp_range, exp_range]), so rows span many magnitudes and a full-size
    batch needs no full-size draw; ``materialise`` builds any rows of it
    exactly, on any device."""
    seqlens = np.asarray(seqlens, dtype=np.int64)
    n_blocks = (seqlens + page - 1) // page
    used = int(n_blocks.sum())
    num_blocks = max(used + spare_blocks, 1)
    perm = permutation(seed, 11, num_blocks)
    slots = []
    k = 0
    for i in range(len(seqlens)):
        j = np.arange(int(seqlens[i]), dtype=np.int64)
        slots.append(perm[k + j // page].astype(np.int64) * page + j % page)
        k += int(n_blocks[i])
    slots = np.concatenate(slots) if slots else np.zeros(0, dtype=np.int64)
    if pad_tokens:
        at = np.sort(randint(seed, 12, pad_tokens, 0, len(slots)))
        slots = np.insert(slots, at, -1)
    n = len(slots)
    exponent = randint(seed, 13, n, -exp_range, exp_range) if n else np.zeros(0, dtype=np.int64)
    base = to_bf16(normal(seed, 14, (base_tokens, h_kv, hd)))
    return CacheWriteInputs(base=base, exponent=exponent.astype(np.int64),
                            slot_mapping=torch.from_numpy(slots.astype(np.int32)),
                            num_blocks=num_blocks, page=page, seqlens=seqlens)


def materialise(inp: CacheWriteInputs, tokens=None, device=None) -> torch.Tensor:
    """bf16 rows of the given tokens (all by default): base row times 2^exponent (exact)."""
    n = len(inp.exponent)
    t = torch.arange(n, dtype=torch.int64) if tokens is None else torch.as_tensor(tokens, dtype=torch.int64)
    base = inp.base.to(device) if device is not None else inp.base
    idx = (t % base.shape[0]).to(base.device)
    f = torch.from_numpy(np.ldexp(1.0, inp.exponent[t.numpy()]).astype(np.float32)).to(base.device)
    return (base[idx].float() * f[:, None, None]).to(torch.bfloat16)


def per_row_scales(seed: int, purpose: int, shape, base: float) -> torch.Tensor:
    """Positive float32 scales, one per cached row: base * 2^u with u uniform in [-2, 2]
    (a seeded stand-in for the amax / 448 of each row)."""
    n = int(np.prod(shape))
    u = uniform(seed, purpose, n).reshape(shape) * 4.0 - 2.0
    return torch.from_numpy((base * np.exp2(u)).astype(np.float32))


def gqa_block_q(seed: int, bs: int, q_len: int, h_q: int, hd: int = 128) -> torch.Tensor:
    """bf16 [bs, q_len, h_q, hd] N(0, 1) queries of a speculative block of q_len tokens."""
    return to_bf16(normal(seed, 31, (bs, q_len, h_q, hd)))


def spec_mask(seed: int, bs: int, q_len: int) -> torch.Tensor:
    """uint8 [bs, q_len, q_len] speculative-decoding mask: each token sees itself and a seeded
    half of the block's other keys (a tree of draft tokens need not be causal)."""
    m = (uniform(seed, 32, bs * q_len * q_len).reshape(bs, q_len, q_len) < 0.5).astype(np.uint8)
    idx = np.arange(q_len)
    m[:, idx, idx] = 1
    return torch.from_numpy(m)


def sink_logits(seed: int, h_q: int) -> torch.Tensor:
    """float32 [h_q] attention-sink logits, uniform in [-2, 6] (the scale of the scaled scores)."""
    return torch.from_numpy((uniform(seed, 33, h_q) * 8.0 - 2.0).astype(np.float32))
