"""fp64 CPU oracle for decode attention over an FP8 (E4M3) paged KV cache.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may
import this package.  The CUDA library never calls it, and it shares no code,
header, table or constant generator with the CUDA library: the two meet only
in the seeded inputs of ``paged_decode_attention_fp8_gb300.synthetic``.

What it computes is the plain definition of softmax attention over the
dequantised cache, in float64, so that a reader can check every function
against the pages by eye:

* ``e4m3_value`` / ``E4M3_TABLE`` -- the OCP E4M3 ("fn") code, all 256
  patterns: sign, 4-bit exponent with bias 7, 3-bit mantissa, no infinity,
  only S.1111.111 is NaN, largest finite 448.  (aiter "Support fp8 KV caches
  and fp8 dots in sparse_mla_fwd on gfx942": the OCP e4m3 vs e4m3fnuz
  distinction; InfiniCore "FP8(E4M3) KV cache support in paged attention",
  Summary: scales are amax/448.)
* ``mla_decode`` -- paged MLA decode, d = 576 (512 latent + 64 RoPE),
  dv = 512, V = the first 512 dims of the same cached row, one KV head,
  page 64 tokens, per-tensor kv_scale, bottom-right causal mask for s_q > 1
  (FlashMLA "update fp8 support": the test shape b, s_q, h_q, h_kv=1, d=576,
  dv=512, causal=True).
* ``sparse_mla_decode`` -- the same with the keys of each query token given
  by a top-k index list into one flat cache, d = dv = 512 rope-free
  (aiter page, Results: 16 heads, rope-free 512, top-k 2048).
* ``gqa_decode`` -- paged GQA decode with separate K and V caches
  [num_blocks, h_kv, page, head_dim] and per-tensor k_scale / v_scale
  (InfiniCore page, Summary: the FP8 paged-attention decode kernel), or
  per-row scales [num_blocks, h_kv, page] (the same page's scale layout);
  ``mla_decode`` takes per-row scales [num_pages, 1, page] the same way.
* ``gqa_decode_ext`` -- the same with the XQA options of the FlashInfer page
  (speculative-decoding block with a mask, sliding window, attention sinks).
* ``partial_attention`` / ``merge_partials`` -- the split-KV algebra: each
  shard publishes (max, sum of exponentials, weighted sum) and the merge
  rescales by exp(m_s - M) (InfiniCore page, split-kv commit: "log2-domain
  merge, standard flash-decoding"; the zero-length-row commit: an empty shard
  is the neutral element m=-inf, l=0, acc=0).
* ``schedule`` -- the deterministic page-range partition the metadata kernel
  emits, restated independently for a bit-exact comparison.

Conventions that the pages leave open, and the reading taken:
* LSE is the natural log of the sum of exp(scaled score), one float per
  (batch, query token, head).
* Causal alignment is bottom-right: query token i of s_q sees keys
  j < s_k - s_q + i + 1.
* A row with no visible key (empty cache, causal cut, all indices -1) has
  output 0 and LSE -inf (InfiniCore zero-length-row commit; FlashInfer
  "add xqa fp8 mha and fp8 kv cache", review of masked rows: a fully masked
  row must give zeros, not the mean of V).
* Bytes of a page past the sequence length, and pages the block table does
  not reference, are never read.
* GQA head h reads KV head h // (h_q // h_kv).
"""

from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------- E4M3 ----


def e4m3_value(code: int) -> float:
    """Value of one E4M3 ("fn") byte, from its bit fields."""
    code = int(code) & 0xFF
    sign = -1.0 if code >> 7 else 1.0
    exponent = (code >> 3) & 0xF
    mantissa = code & 0x7
    if exponent == 0xF and mantissa == 0x7:
        return math.nan
    if exponent == 0:                       # subnormal: (m / 8) * 2^(1 - 7)
        return sign * (mantissa / 8.0) * 2.0 ** -6
    return sign * (1.0 + mantissa / 8.0) * 2.0 ** (exponent - 7)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of an array of E4M3 bytes."""
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def as_float64(x) -> np.ndarray:
    """float64 copy of a numpy array or a (CPU) torch tensor, exact for bf16."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().numpy()
    return np.asarray(x, dtype=np.float64)


def as_int64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.asarray(x, dtype=np.int64)


def as_bytes(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if x.dtype != __import__("torch").uint8:
            x = x.view(__import__("torch").uint8)
        x = x.numpy()
    return np.asarray(x, dtype=np.uint8)


# ------------------------------------------------------- softmax rows ----


def softmax_attention(scores: np.ndarray, values: np.ndarray):
    """Attention of one row: softmax(scores) @ values and its natural-log LSE.

    scores: [n] float64, values: [n, dv].  n == 0 gives (zeros, -inf).
    """
    dv = values.shape[1]
    if scores.shape[0] == 0:
        return np.zeros(dv), -math.inf
    m = np.max(scores)
    e = np.exp(scores - m)
    total = np.sum(e)
    lse = m + math.log(total)
    return (e / total) @ values, lse


def partial_attention(scores: np.ndarray, values: np.ndarray):
    """One shard's (m, l, acc): max score, sum of exp(s - m), sum of exp(s - m) v."""
    dv = values.shape[1]
    if scores.shape[0] == 0:
        return -math.inf, 0.0, np.zeros(dv)
    m = float(np.max(scores))
    e = np.exp(scores - m)
    return m, float(np.sum(e)), e @ values


def merge_partials(parts):
    """Merge shard triples: M = max m_s, L = sum l_s e^(m_s - M),
    out = sum acc_s e^(m_s - M) / L, lse = M + ln L.  Empty shards drop out."""
    live = [(m, l, a) for (m, l, a) in parts if m != -math.inf]
    dv = parts[0][2].shape[0]
    if not live:
        return np.zeros(dv), -math.inf
    big_m = max(m for m, _, _ in live)
    big_l = sum(l * math.exp(m - big_m) for m, l, _ in live)
    acc = sum(a * math.exp(m - big_m) for m, _, a in live)
    return acc / big_l, big_m + math.log(big_l)


# ------------------------------------------------------------ dense MLA ----


def mla_visible_keys(s_k: int, s_q: int, i: int, causal: bool) -> int:
    """Number of keys query token i sees (bottom-right causal alignment)."""
    return max(0, s_k - s_q + i + 1) if causal else s_k


def key_scales(scale, pages, head: int, s_k: int):
    """The dequantisation scale of each of a sequence's s_k keys.

    ``scale`` is one float (per tensor) or an array [num_blocks, h_kv, page]
    with one float per cached row (InfiniCore page, Summary: FP8 caches carry
    scales of shape [num_blocks, num_kv_heads, block_size]); key j of the
    sequence lives in block pages[j // page] at offset j % page.  Returns a
    float or a column [s_k, 1]."""
    if np.ndim(scale) == 0:
        return float(scale)
    sc = as_float64(scale)
    if not pages:
        return np.zeros((0, 1))
    return np.concatenate([sc[p, head] for p in pages])[:s_k][:, None]


def mla_gather_keys(kv_cache, block_table_row, s_k: int, kv_scale, page: int = 64):
    """Dequantised keys [s_k, d] of one sequence, read page by page.  kv_scale:
    one float, or per cached row [num_pages, 1, page]."""
    cache = as_bytes(kv_cache)
    n_pages = (s_k + page - 1) // page
    pages = [int(block_table_row[p]) for p in range(n_pages)]
    rows = [cache[p] for p in pages]
    if not rows:
        return np.zeros((0, cache.shape[-1]))
    keys = np.concatenate(rows, axis=0)[:s_k]
    return e4m3_decode(keys) * key_scales(kv_scale, pages, 0, s_k)


def mla_decode(q, kv_cache, block_table, seqlens, kv_scale, softmax_scale, causal,
               dv: int = 512, page: int = 64, batches=None):
    """Paged MLA decode.

    q [b, s_q, h_q, d] (bf16 values), kv_cache [num_pages, page, d] E4M3 bytes,
    block_table [b, max_pages], seqlens [b].  Returns out [b, s_q, h_q, dv]
    and lse [b, s_q, h_q] in float64.  ``batches`` restricts the work to some
    sequences (the others stay 0 / NaN).
    """
    q = as_float64(q)
    bt = as_int64(block_table)
    sl = as_int64(seqlens)
    b, s_q, h_q, d = q.shape
    out = np.zeros((b, s_q, h_q, dv))
    lse = np.full((b, s_q, h_q), np.nan)
    for bi in (range(b) if batches is None else batches):
        s_k = int(sl[bi])
        keys = mla_gather_keys(kv_cache, bt[bi], s_k, kv_scale, page)
        values = keys[:, :dv]
        scores = (q[bi].reshape(s_q * h_q, d) @ keys.T) * float(softmax_scale)
        scores = scores.reshape(s_q, h_q, s_k)
        for i in range(s_q):
            n_vis = mla_visible_keys(s_k, s_q, i, causal)
            for h in range(h_q):
                out[bi, i, h], lse[bi, i, h] = softmax_attention(scores[i, h, :n_vis],
                                                                 values[:n_vis])
    return out, lse


# ----------------------------------------------------------- sparse MLA ----


def sparse_mla_decode(q, kv_cache, topk_idx, kv_scale, softmax_scale, tokens=None):
    """Top-k sparse MLA decode: token t attends to the rows topk_idx[t] (-1 skipped).

    q [s_q, h_q, d], kv_cache [num_tokens, d] E4M3 bytes, V = K (d = dv).
    """
    q = as_float64(q)
    cache = as_bytes(kv_cache)
    idx = as_int64(topk_idx)
    s_q, h_q, d = q.shape
    out = np.zeros((s_q, h_q, d))
    lse = np.full((s_q, h_q), np.nan)
    for t in (range(s_q) if tokens is None else tokens):
        rows = idx[t][idx[t] != -1]
        keys = e4m3_decode(cache[rows]) * float(kv_scale)
        scores = (q[t] @ keys.T) * float(softmax_scale)
        for h in range(h_q):
            out[t, h], lse[t, h] = softmax_attention(scores[h], keys)
    return out, lse


# ------------------------------------------------------------------ GQA ----


def gqa_decode(q, k_cache, v_cache, block_table, seqlens, k_scale, v_scale, softmax_scale,
               batches=None):
    """Paged GQA decode.  q [bs, h_q, hd]; caches [num_blocks, h_kv, page, hd];
    k_scale / v_scale one float each, or per cached row [num_blocks, h_kv, page]."""
    q = as_float64(q)
    kc = as_bytes(k_cache)
    vc = as_bytes(v_cache)
    bt = as_int64(block_table)
    sl = as_int64(seqlens)
    bs, h_q, hd = q.shape
    _, h_kv, page, _ = kc.shape
    group = h_q // h_kv
    out = np.zeros((bs, h_q, hd))
    lse = np.full((bs, h_q), np.nan)
    for bi in (range(bs) if batches is None else batches):
        s_k = int(sl[bi])
        for kvh in range(h_kv):
            keys, vals = gqa_gather(kc, vc, bt[bi], s_k, kvh, k_scale, v_scale)
            for h in range(kvh * group, (kvh + 1) * group):
                scores = (keys @ q[bi, h]) * float(softmax_scale)
                out[bi, h], lse[bi, h] = softmax_attention(scores, vals)
    return out, lse


def gqa_gather(kc, vc, block_table_row, s_k: int, kvh: int, k_scale, v_scale):
    """Dequantised keys and values [s_k, hd] of one sequence and KV head."""
    page, hd = kc.shape[2], kc.shape[3]
    pages = [int(block_table_row[p]) for p in range((s_k + page - 1) // page)]
    if not pages:
        return np.zeros((0, hd)), np.zeros((0, hd))
    keys = e4m3_decode(np.concatenate([kc[p, kvh] for p in pages])[:s_k]) * key_scales(k_scale, pages, kvh, s_k)
    vals = e4m3_decode(np.concatenate([vc[p, kvh] for p in pages])[:s_k]) * key_scales(v_scale, pages, kvh, s_k)
    return keys, vals


def spec_visible(s_k: int, q_len: int, i: int, mask_row=None, window: int = 0) -> np.ndarray:
    """Keys query token i of a speculative block sees (FlashInfer "add xqa fp8
    mha and fp8 kv cache": the XQA mask gate).  The q_len query tokens are the
    last q_len cache positions, token i at p = s_k - q_len + i.  Keys before
    the block are always visible; key s_k - q_len + c of the block is visible
    iff mask_row[c] (no mask: c <= i, the causal case).  A sliding window
    W > 0 further keeps only keys with p - j < W.  Returns a bool [s_k]."""
    j = np.arange(s_k)
    start = s_k - q_len
    vis = j < start
    c = j - start
    in_block = (c >= 0) & (c < q_len)
    if mask_row is None:
        vis |= in_block & (c <= i)
    else:
        m = np.asarray(mask_row, dtype=bool)
        vis |= in_block & m[np.clip(c, 0, q_len - 1)]
    if window > 0:
        vis &= (start + i) - j < window
    return vis


def gqa_decode_ext(q, k_cache, v_cache, block_table, seqlens, k_scale, v_scale, softmax_scale,
                   spec_mask=None, window: int = 0, sinks=None):
    """Paged GQA decode with the XQA options of the FlashInfer page: a block of
    q_len query tokens per sequence (q [bs, q_len, h_q, hd]) under a
    speculative-decoding mask spec_mask [bs, q_len, q_len] (None: causal), a
    sliding window (0: off) and attention sinks (one logit per query head,
    None: off).

    With a sink s_h, head h's softmax denominator gains e^{s_h} (a key with no
    value): out = sum_j e^{s_j} v_j / (sum_j e^{s_j} + e^{s_h}) and
    lse = ln(sum_j e^{s_j} + e^{s_h}).  A row that sees no key has out = 0 and
    lse = s_h (-inf without a sink) -- zeros, not the mean of V (FlashInfer
    page, review of masked rows).  Returns out [bs, q_len, h_q, hd] and lse
    [bs, q_len, h_q]."""
    q = as_float64(q)
    kc = as_bytes(k_cache)
    vc = as_bytes(v_cache)
    bt = as_int64(block_table)
    sl = as_int64(seqlens)
    bs, q_len, h_q, hd = q.shape
    h_kv = kc.shape[1]
    group = h_q // h_kv
    sk = None if sinks is None else as_float64(sinks)
    out = np.zeros((bs, q_len, h_q, hd))
    lse = np.full((bs, q_len, h_q), np.nan)
    for bi in range(bs):
        s_k = int(sl[bi])
        for kvh in range(h_kv):
            keys, vals = gqa_gather(kc, vc, bt[bi], s_k, kvh, k_scale, v_scale)
            for i in range(q_len):
                vis = spec_visible(s_k, q_len, i, None if spec_mask is None else as_int64(spec_mask)[bi, i],
                                   window)
                for h in range(kvh * group, (kvh + 1) * group):
                    scores = (keys[vis] @ q[bi, i, h]) * float(softmax_scale)
                    o, l = softmax_attention(scores, vals[vis])
                    if sk is not None and sk[h] != -math.inf:
                        # the sink joins the denominator (shifted by the larger exponent)
                        m = max(l, sk[h])
                        w_keys = math.exp(l - m) if l != -math.inf else 0.0
                        denom = w_keys + math.exp(sk[h] - m)
                        o = o * (w_keys / denom)
                        l = m + math.log(denom)
                    out[bi, i, h], lse[bi, i, h] = o, l
    return out, lse


# ------------------------------------------------------------ scheduler ----

SCHED_PAGE = 64
SCHED_FIXED_COST = 4      # pages-equivalent cost of one (sequence, unit) segment
SCHED_FIELDS = 8


def schedule(seqlens, num_units: int, force_splits: int = 0, page: int = SCHED_PAGE,
             fixed_cost: int = SCHED_FIXED_COST):
    """Page-range partition of a batch over ``num_units`` work units.

    Returns (tile_sched [num_units, 8] int32, num_splits [b + 1] int32).
    Unit u covers the flattened (sequence, page) positions from
    (b_begin, page_begin) up to but excluding (b_end, page_end); field 4 is
    the index, among the pieces sequence b_begin is cut into, of the unit's
    first piece.  num_splits is the prefix sum of the number of pieces of
    each sequence.

    Balanced rule (force_splits == 0): lay the sequences on one cost line,
    each non-empty sequence taking (pages + fixed_cost) positions; unit u
    gets positions [floor(u W / U), floor((u + 1) W / U)) of the W in all.
    A position maps to page max(0, offset - fixed_cost) of its sequence, so
    a sequence's first fixed_cost positions stand for its page 0.  Units
    whose interval holds no page are empty.  Forced rule (force_splits = k):
    sequence i is cut into c = min(k, n_i) chunks, chunk j being pages
    [floor(j n_i / c), floor((j + 1) n_i / c)), one unit per chunk in order.
    """
    sl = as_int64(seqlens)
    b = sl.shape[0]
    n = [(int(s) + page - 1) // page if s > 0 else 0 for s in sl]
    sched = np.zeros((num_units, SCHED_FIELDS), dtype=np.int32)
    count = [0] * b

    if force_splits > 0:
        chunks = []
        for i in range(b):
            c = min(force_splits, n[i])
            for j in range(c):
                chunks.append((i, (j * n[i]) // c, (j + 1) * n[i] // c, j))
        if len(chunks) > num_units:
            raise ValueError("more chunks than units")
        for u in range(num_units):
            if u < len(chunks):
                i, p0, p1, j = chunks[u]
                # a chunk that ends a sequence is written as (i + 1, 0)
                end = (i + 1, 0) if p1 == n[i] else (i, p1)
                sched[u] = [i, p0, end[0], end[1], j, 0, 0, 0]
                count[i] += 1
            else:
                sched[u] = [b, 0, b, 0, 0, 0, 0, 0]
    else:
        cost = [x + fixed_cost if x > 0 else 0 for x in n]
        begin = [0] * (b + 1)
        for i in range(b):
            begin[i + 1] = begin[i] + cost[i]
        total = begin[b]

        def position(x):
            for i in range(b):
                if cost[i] > 0 and begin[i] <= x < begin[i] + cost[i]:
                    return (i, max(0, x - begin[i] - fixed_cost))
            return (b, 0)

        starts = [position(u * total // num_units) for u in range(num_units)] + [(b, 0)]
        for u in range(num_units):
            (bs, ps), (be, pe) = starts[u], starts[u + 1]
            nonempty = (bs, ps) < (be, pe)
            first = 0
            if nonempty and ps > 0:
                first = sum(1 for v in range(u + 1)
                            if starts[v][0] == bs and starts[v][1] > 0 and starts[v] < starts[v + 1])
            sched[u] = [bs, ps, be, pe, first, 0, 0, 0]
            if nonempty:
                for i in range(bs, min(be, b - 1) + 1):
                    lo = ps if i == bs else 0
                    hi = pe if i == be else n[i]
                    if hi > lo:
                        count[i] += 1

    num_splits = np.zeros(b + 1, dtype=np.int32)
    num_splits[1:] = np.cumsum(count)
    return sched, num_splits


def unit_segments(sched_row, seqlens, page: int = SCHED_PAGE):
    """(sequence, first page, end page, split index) segments of one unit."""
    sl = as_int64(seqlens)
    b0, p0, b1, p1, first = (int(x) for x in sched_row[:5])
    segs = []
    for bi in range(b0, min(b1, sl.shape[0] - 1) + 1):
        n_b = (int(sl[bi]) + page - 1) // page
        lo = p0 if bi == b0 else 0
        hi = p1 if bi == b1 else n_b
        if hi > lo:
            segs.append((bi, lo, hi, first if bi == b0 else 0))
    return segs
