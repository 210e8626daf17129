"""Pins of the oracle's per-row KV scales ([num_blocks, h_kv, page], the
scale layout of the InfiniCore FP8 KV-cache page) against facts that do not
come from the oracle's page walk:

* a per-row array that holds the per-tensor scale everywhere gives the
  per-tensor result bit for bit (GQA and dense MLA);
* brute force: keys and values rebuilt token by token from the block table
  with their own row's scale, then a plain softmax;
* round trip: rows quantised on write with per-row scales (the cache-write
  oracle) and decoded with those scales stay within E4M3's rounding of the
  attention over the unquantised values, and beat one per-tensor scale when
  row magnitudes differ widely.
"""

import math

import numpy as np

import oracle
from oracle.attention import e4m3_decode
from oracle.cache_write import paged_cache_write
from paged_decode_attention_fp8_gb300 import synthetic as syn


def _row_scales(seed, shape):
    # positive per-row scales spanning 2^-3 .. 2^3
    return np.exp2(syn.uniform(seed, 40, int(np.prod(shape))) * 6.0 - 3.0).reshape(shape).astype(np.float32)


def test_constant_row_scales_equal_per_tensor_gqa():
    inp = syn.gqa_inputs(31, 3, [40, 1, 70], h_q=8, h_kv=2, hd=32, spare_blocks=2)
    nb, h_kv, page, _ = inp.k_cache.shape
    ks = np.full((nb, h_kv, page), inp.k_scale, dtype=np.float64)
    vs = np.full((nb, h_kv, page), inp.v_scale, dtype=np.float64)
    a = oracle.gqa_decode(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.seqlens, inp.k_scale,
                          inp.v_scale, inp.softmax_scale)
    b = oracle.gqa_decode(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.seqlens, ks, vs,
                          inp.softmax_scale)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_constant_row_scales_equal_per_tensor_mla():
    inp = syn.mla_inputs(32, 2, 2, 8, [100, 30], causal=True, spare_pages=3)
    num_pages = inp.kv_cache.shape[0]
    sc = np.full((num_pages, 1, 64), inp.kv_scale, dtype=np.float64)
    a = oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens, inp.kv_scale, inp.softmax_scale, True)
    b = oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens, sc, inp.softmax_scale, True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def _softmax_rows(scores, vals):
    m = max(scores)
    w = [math.exp(s - m) for s in scores]
    tot = math.fsum(w)
    out = np.array([math.fsum(w[j] * vals[j][c] for j in range(len(w))) / tot for c in range(len(vals[0]))])
    return out, m + math.log(tot)


def test_gqa_row_scales_brute_force():
    inp = syn.gqa_inputs(33, 2, [37, 20], h_q=4, h_kv=2, hd=16, spare_blocks=3)
    nb, h_kv, page, hd = inp.k_cache.shape
    ks, vs = _row_scales(33, (nb, h_kv, page)), _row_scales(34, (nb, h_kv, page))
    out, lse = oracle.gqa_decode(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.seqlens, ks, vs,
                                 inp.softmax_scale)
    q = inp.q.float().numpy().astype(np.float64)
    kc, vc = inp.k_cache.numpy(), inp.v_cache.numpy()
    bt = inp.block_table.numpy()
    for b, s_k in enumerate(inp.seqlens.tolist()):
        for h in range(4):
            kvh = h // 2
            keys, vals = [], []
            for j in range(s_k):
                blk, off = int(bt[b, j // page]), j % page
                keys.append([float(ks[blk, kvh, off]) * float(e4m3_decode(c)) for c in kc[blk, kvh, off]])
                vals.append([float(vs[blk, kvh, off]) * float(e4m3_decode(c)) for c in vc[blk, kvh, off]])
            scores = [math.fsum(q[b, h, c] * keys[j][c] for c in range(hd)) * inp.softmax_scale
                      for j in range(s_k)]
            o, l = _softmax_rows(scores, vals)
            assert np.allclose(out[b, h], o, rtol=1e-12, atol=1e-14)
            assert abs(lse[b, h] - l) < 1e-12


def test_mla_row_scales_brute_force():
    inp = syn.mla_inputs(35, 2, 1, 2, [70, 9], causal=False, spare_pages=2)
    num_pages = inp.kv_cache.shape[0]
    sc = _row_scales(35, (num_pages, 1, 64))
    out, lse = oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens, sc, inp.softmax_scale, False)
    q = inp.q.float().numpy().astype(np.float64)
    cache = inp.kv_cache.numpy()
    bt = inp.block_table.numpy()
    for b, s_k in enumerate(inp.seqlens.tolist()):
        rows = []
        for j in range(s_k):
            blk, off = int(bt[b, j // 64]), j % 64
            rows.append(e4m3_decode(cache[blk, off]) * float(sc[blk, 0, off]))
        keys = np.array(rows)
        for h in range(2):
            scores = [math.fsum(q[b, 0, h] * keys[j]) * inp.softmax_scale for j in range(s_k)]
            o, l = _softmax_rows(scores, keys[:, :512].tolist())
            assert np.allclose(out[b, 0, h], o, rtol=1e-12, atol=1e-14)
            assert abs(lse[b, 0, h] - l) < 1e-12


def test_round_trip_through_the_cache_write():
    # V rows of a whole sequence sit at very different magnitudes (2^8, 2^-8, 1);
    # quantised on write with per-row scales and read back by the decode, every
    # (sequence, head) output stays within E4M3's rounding of the exact attention
    # over the unquantised rows, while one per-tensor scale loses the small sequence
    seqlens = [45, 130, 16]
    h_kv, hd, page, h_q = 2, 64, 16, 4
    kin = syn.cache_write_inputs(36, seqlens, h_kv=h_kv, hd=hd, page=page, base_tokens=191, exp_range=0)
    vin = syn.cache_write_inputs(37, seqlens, h_kv=h_kv, hd=hd, page=page, base_tokens=191, exp_range=0)
    vin.exponent = np.concatenate([np.full(n, e) for n, e in zip(seqlens, (8, -8, 0))]).astype(np.int64)
    k = syn.materialise(kin)
    v = syn.materialise(vin)
    slots = kin.slot_mapping.numpy().astype(np.int64)
    nb = kin.num_blocks
    # block table from the slot of each page's first token
    starts = np.cumsum([0] + seqlens[:-1])
    max_blocks = max((n + page - 1) // page for n in seqlens)
    bt = np.zeros((len(seqlens), max_blocks), dtype=np.int32)
    for i, n in enumerate(seqlens):
        for p in range((n + page - 1) // page):
            bt[i, p] = slots[starts[i] + p * page] // page
    q = syn.to_bf16(syn.normal(38, 0, (len(seqlens), h_q, hd)) * 0.2)
    softmax_scale = 1.0 / math.sqrt(hd)
    zero = np.zeros((nb, h_kv, page, hd), dtype=np.uint8)
    ones = np.ones((nb, h_kv, page), dtype=np.float32)
    kc, ks = paged_cache_write(k, slots, zero, page, token_scales=ones)
    vc, vs = paged_cache_write(v, slots, zero, page, token_scales=ones)
    out, lse = oracle.gqa_decode(q, kc, vc, bt, np.array(seqlens), ks, vs, softmax_scale)
    kt = float(np.float32(np.abs(k.float().numpy()).max() / 448.0))
    vt = float(np.float32(np.abs(v.float().numpy()).max() / 448.0))
    kc1, _ = paged_cache_write(k, slots, zero, page, tensor_scale=kt)
    vc1, _ = paged_cache_write(v, slots, zero, page, tensor_scale=vt)
    out1, _ = oracle.gqa_decode(q, kc1, vc1, bt, np.array(seqlens), kt, vt, softmax_scale)
    kf, vf, qf = (t.float().numpy().astype(np.float64) for t in (k, v, q))
    ref = np.zeros_like(out)
    ref_lse = np.zeros_like(lse)
    for i, n in enumerate(seqlens):
        rows = slice(starts[i], starts[i] + n)
        for h in range(h_q):
            kvh = h // (h_q // h_kv)
            ref[i, h], ref_lse[i, h] = oracle.softmax_attention(kf[rows, kvh] @ qf[i, h] * softmax_scale,
                                                                vf[rows, kvh])
    rel = np.linalg.norm(out - ref, axis=-1) / np.linalg.norm(ref, axis=-1)
    rel1 = np.linalg.norm(out1 - ref, axis=-1) / np.linalg.norm(ref, axis=-1)
    assert 0 < rel.max() < 0.05               # E4M3 keeps ~2^-4 relative per element
    assert rel1[1].max() > 0.2                # the 2^-8 sequence under one per-tensor scale
    assert np.max(np.abs(lse - ref_lse)) < 0.01
