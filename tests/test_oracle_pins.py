"""Pins of the fp64 oracle against facts that do not come from the oracle.

* E4M3 decoding: the page-fixed points (largest value 448, the NaN code),
  every code against torch's own float8_e4m3fn decoding, monotonicity.
* Closed forms: all-equal scores give the mean of V; the peaky case of the
  aiter sparse_mla_fwd page (one key +9 above 2047, a fifth of the output in
  the tail); a single key returns its own value.
* Brute force: a second, loop-only implementation with torch's decoding,
  correctly rounded dot products (math.fsum) and 50-digit decimal exp/ln.
* Invariants: split/merge equals the direct result (InfiniCore split-kv
  commit), physical page relabelling leaves the result bit-identical.
"""

import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import oracle
from paged_decode_attention_fp8_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ----------------------------------------------------------------- E4M3 ----


def test_e4m3_page_pins():
    for code, value in _golden_rows("e4m3_pins.txt"):
        got = oracle.e4m3_value(int(code, 16))
        if value == "nan":
            assert math.isnan(got), code
        else:
            assert got == float(value), (code, got, value)
            assert math.copysign(1.0, got) == math.copysign(1.0, float(value)), code


def test_e4m3_table_matches_torch_for_all_codes():
    torch_vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    ref = torch_vals.numpy()
    for c in range(256):
        if math.isnan(ref[c]):
            assert math.isnan(oracle.E4M3_TABLE[c])
        else:
            assert oracle.E4M3_TABLE[c] == ref[c], c
    assert int(np.isnan(oracle.E4M3_TABLE).sum()) == 2


def test_e4m3_monotone_and_symmetric():
    pos = oracle.E4M3_TABLE[0:0x7F]
    assert np.all(np.diff(pos) > 0)
    assert pos[-1] == 448.0
    for c in range(0x7F):
        assert oracle.E4M3_TABLE[c | 0x80] == -oracle.E4M3_TABLE[c]


def test_e4m3_encode_decode_round_trip():
    # every finite code survives decode -> the input generator's encoder
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    back = syn.to_e4m3_bytes(vals, 1.0)
    assert np.array_equal(back, codes)


def test_amax_scale_puts_largest_at_448():
    x = syn.normal(5, 1, (1000,))
    scale = syn.per_tensor_scale(x)
    enc = syn.to_e4m3_bytes(x, scale)
    dec = oracle.e4m3_decode(enc)
    assert np.max(np.abs(dec)) == 448.0
    assert abs(oracle.e4m3_decode(enc[np.argmax(np.abs(x))])) == 448.0


# --------------------------------------------------------- closed forms ----


def _tiny_mla(seed=1, b=2, s_q=1, h_q=4, seqlens=(70, 5), causal=False, spare=3):
    return syn.mla_inputs(seed, b, s_q, h_q, list(seqlens), causal=causal, spare_pages=spare)


def test_equal_scores_give_mean_of_v():
    inp = _tiny_mla(seqlens=(130, 64))
    q = torch.zeros_like(inp.q)
    out, lse = oracle.mla_decode(q, inp.kv_cache, inp.block_table, inp.seqlens,
                                 inp.kv_scale, inp.softmax_scale, False)
    for bi, s_k in enumerate(inp.seqlens.tolist()):
        keys = oracle.attention.mla_gather_keys(inp.kv_cache, inp.block_table[bi].numpy(),
                                                s_k, inp.kv_scale)
        mean_v = keys[:, :512].mean(axis=0)
        assert np.allclose(out[bi, 0], mean_v[None, :], rtol=0, atol=1e-12)
        assert np.allclose(lse[bi], math.log(s_k), rtol=0, atol=1e-12)


def test_peaky_closed_form_and_page_fifth():
    margin, n_tail, share, tol = (float(x) for x in _golden_rows("peaky_tail.txt")[0])
    n_tail = int(n_tail)
    d = 512
    rng = np.random.default_rng(0)
    z = rng.standard_normal(256)
    tail_vals = rng.standard_normal((n_tail, 256))
    # bytes: key 0 has 448 in dim 0 and z (encoded) in dims 256+; tails are 0 on [0, 256)
    kv_scale = 2.0 ** -6                      # 448 * 2^-6 = 7 exactly
    cache = np.zeros((n_tail + 1, d), dtype=np.uint8)
    cache[0, 0] = 0x7E
    cache[0, 256:] = syn.to_e4m3_bytes(z, kv_scale)
    cache[1:, 256:] = syn.to_e4m3_bytes(tail_vals, kv_scale)
    q = np.zeros((1, 1, d))
    q[0, 0, 0] = margin / 7.0
    q[0, 0, 1:256] = rng.standard_normal(255)
    idx = np.arange(n_tail + 1, dtype=np.int32)[None, :]
    out, lse = oracle.sparse_mla_decode(q, cache, idx, kv_scale, 1.0)
    w0 = 1.0 / (1.0 + n_tail * math.exp(-margin))
    assert abs(lse[0, 0] - (margin + math.log(1.0 + n_tail * math.exp(-margin)))) < 1e-12
    v = oracle.e4m3_decode(cache) * kv_scale
    expect = w0 * v[0] + (1.0 - w0) * v[1:].mean(axis=0)
    assert np.allclose(out[0, 0], expect, rtol=0, atol=1e-12)
    assert abs((1.0 - w0) - share) < tol          # "a fifth of the output"
    assert abs(w0 - 0.798325) < 1e-5


def test_single_key():
    inp = _tiny_mla(seqlens=(1, 1), h_q=3)
    out, lse = oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens,
                                 inp.kv_scale, inp.softmax_scale, False)
    for bi in range(2):
        k = oracle.attention.mla_gather_keys(inp.kv_cache, inp.block_table[bi].numpy(), 1,
                                             inp.kv_scale)
        q = inp.q[bi, 0].double().numpy()
        assert np.array_equal(out[bi, 0], np.repeat(k[:, :512], 3, axis=0))
        assert np.allclose(lse[bi, 0], q @ k[0] * inp.softmax_scale, rtol=0, atol=1e-12)


def test_empty_and_fully_masked_rows():
    inp = _tiny_mla(seqlens=(0, 1), s_q=2, causal=True)
    out, lse = oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens,
                                 inp.kv_scale, inp.softmax_scale, True)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    # s_k = 1, s_q = 2, causal: token 0 sees no key, token 1 sees key 0
    assert np.all(out[1, 0] == 0) and np.all(np.isneginf(lse[1, 0]))
    assert np.all(np.isfinite(lse[1, 1]))


def test_causal_token_equals_shorter_cache():
    inp = _tiny_mla(seqlens=(100, 65), s_q=2, causal=True)
    out_c, lse_c = oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens,
                                     inp.kv_scale, inp.softmax_scale, True)
    shorter = inp.seqlens - 1
    out_s, lse_s = oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, shorter,
                                     inp.kv_scale, inp.softmax_scale, False)
    assert np.array_equal(out_c[:, 0], out_s[:, 0]) and np.array_equal(lse_c[:, 0], lse_s[:, 0])
    out_f, lse_f = oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens,
                                     inp.kv_scale, inp.softmax_scale, False)
    assert np.array_equal(out_c[:, 1], out_f[:, 1])


def test_gqa_groups_share_kv_head():
    inp = syn.gqa_inputs(3, 2, [40, 17], h_q=8, h_kv=2, hd=16, page=16, spare_blocks=2)
    out, lse = oracle.gqa_decode(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.seqlens,
                                 inp.k_scale, inp.v_scale, inp.softmax_scale)
    # identical queries in one group give identical rows
    q2 = inp.q.clone()
    q2[:, 1] = q2[:, 0]
    out2, _ = oracle.gqa_decode(q2, inp.k_cache, inp.v_cache, inp.block_table, inp.seqlens,
                                inp.k_scale, inp.v_scale, inp.softmax_scale)
    assert np.array_equal(out2[:, 0], out2[:, 1])
    # ... but heads of different groups read different caches
    q3 = inp.q.clone()
    q3[:, 4] = q3[:, 0]
    out3, _ = oracle.gqa_decode(q3, inp.k_cache, inp.v_cache, inp.block_table, inp.seqlens,
                                inp.k_scale, inp.v_scale, inp.softmax_scale)
    assert not np.allclose(out3[:, 0], out3[:, 4])


# ----------------------------------------------------------- brute force ----

getcontext().prec = 50


def _torch_decode(byte):
    return torch.tensor([int(byte)], dtype=torch.uint8).view(torch.float8_e4m3fn).double().item()


def _brute_rows(q_rows, keys, values, scale):
    """Loop-only softmax attention with 50-digit exp / ln.  keys, values: lists of lists."""
    results = []
    for q in q_rows:
        scores = [math.fsum(qi * ki for qi, ki in zip(q, k)) * scale for k in keys]
        if not scores:
            results.append((None, None))
            continue
        m = max(scores)
        ex = [Decimal(s - m).exp() for s in scores]
        tot = sum(ex)
        out = [float(sum(e * Decimal(v[c]) for e, v in zip(ex, values)) / tot)
               for c in range(len(values[0]))]
        results.append((out, float(Decimal(m) + tot.ln())))
    return results


def test_brute_force_mla_paged_causal():
    inp = syn.mla_inputs(11, 2, 2, 2, [70, 9], causal=True, spare_pages=2)
    out, lse = oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens,
                                 inp.kv_scale, inp.softmax_scale, True)
    cache = inp.kv_cache.numpy()
    bt = inp.block_table.numpy()
    for bi, s_k in enumerate(inp.seqlens.tolist()):
        keys = []
        for j in range(s_k):
            row = cache[bt[bi, j // 64], j % 64]
            keys.append([_torch_decode(x) * inp.kv_scale for x in row])
        for i in range(2):
            vis = s_k - 2 + i + 1
            q_rows = [inp.q[bi, i, h].double().tolist() for h in range(2)]
            res = _brute_rows(q_rows, keys[:vis], [k[:512] for k in keys[:vis]],
                              inp.softmax_scale)
            for h, (o, l) in enumerate(res):
                assert np.allclose(out[bi, i, h], o, rtol=1e-12, atol=1e-14)
                assert abs(lse[bi, i, h] - l) < 1e-12


def test_brute_force_sparse_with_skips():
    inp = syn.sparse_inputs(12, 2, h_q=2, num_tokens=300, topk=40)
    idx = inp.topk_idx.clone()
    idx[0, ::7] = -1
    out, lse = oracle.sparse_mla_decode(inp.q, inp.kv_cache, idx, inp.kv_scale,
                                        inp.softmax_scale)
    cache = inp.kv_cache.numpy()
    for t in range(2):
        rows = [int(r) for r in idx[t].tolist() if r != -1]
        keys = [[_torch_decode(x) * inp.kv_scale for x in cache[r]] for r in rows]
        res = _brute_rows([inp.q[t, h].double().tolist() for h in range(2)], keys, keys,
                          inp.softmax_scale)
        for h, (o, l) in enumerate(res):
            assert np.allclose(out[t, h], o, rtol=1e-12, atol=1e-14)
            assert abs(lse[t, h] - l) < 1e-12


def test_brute_force_gqa():
    inp = syn.gqa_inputs(13, 2, [33, 16], h_q=4, h_kv=2, hd=16, page=16, spare_blocks=2)
    out, lse = oracle.gqa_decode(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.seqlens,
                                 inp.k_scale, inp.v_scale, inp.softmax_scale)
    kc, vc, bt = inp.k_cache.numpy(), inp.v_cache.numpy(), inp.block_table.numpy()
    for bi, s_k in enumerate(inp.seqlens.tolist()):
        for h in range(4):
            kvh = h // 2
            keys = [[_torch_decode(x) * inp.k_scale for x in kc[bt[bi, j // 16], kvh, j % 16]]
                    for j in range(s_k)]
            vals = [[_torch_decode(x) * inp.v_scale for x in vc[bt[bi, j // 16], kvh, j % 16]]
                    for j in range(s_k)]
            (o, l), = _brute_rows([inp.q[bi, h].double().tolist()], keys, vals,
                                  inp.softmax_scale)
            assert np.allclose(out[bi, h], o, rtol=1e-12, atol=1e-14)
            assert abs(lse[bi, h] - l) < 1e-12


# ------------------------------------------------------------ invariants ----


def test_split_merge_equals_direct_300_cases():
    rng = np.random.default_rng(1)
    for case in range(300):
        n = int(rng.integers(1, 200))
        s = rng.standard_normal(n) * rng.uniform(0.1, 20)
        v = rng.standard_normal((n, 8))
        direct, lse = oracle.softmax_attention(s, v)
        cuts = np.sort(rng.integers(0, n + 1, size=int(rng.integers(0, 6))))
        bounds = [0, *cuts.tolist(), n]
        parts = [oracle.partial_attention(s[a:e], v[a:e]) for a, e in zip(bounds, bounds[1:])]
        merged, mlse = oracle.merge_partials(parts)
        assert np.allclose(merged, direct, rtol=1e-12, atol=1e-13), case
        assert abs(mlse - lse) < 1e-12 * max(1.0, abs(lse)), case
    # all shards empty -> zeros and -inf
    out, lse = oracle.merge_partials([oracle.partial_attention(np.zeros(0), np.zeros((0, 4)))] * 3)
    assert np.all(out == 0) and lse == -math.inf


def test_page_relabelling_is_bit_identical():
    inp = _tiny_mla(seqlens=(200, 64), h_q=2, spare=5)
    base = oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens,
                             inp.kv_scale, inp.softmax_scale, False)
    num_pages = inp.kv_cache.shape[0]
    perm = np.random.default_rng(2).permutation(num_pages)
    new_cache = np.empty_like(inp.kv_cache.numpy())
    new_cache[perm] = inp.kv_cache.numpy()
    new_bt = perm[inp.block_table.numpy()]
    moved = oracle.mla_decode(inp.q, new_cache, new_bt, inp.seqlens,
                              inp.kv_scale, inp.softmax_scale, False)
    assert np.array_equal(base[0], moved[0]) and np.array_equal(base[1], moved[1])


def test_poisoned_slots_are_never_read():
    inp = _tiny_mla(seqlens=(70, 5), h_q=2, spare=3)
    out, lse = oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens,
                                 inp.kv_scale, inp.softmax_scale, False)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    # the generator did poison: the tail of each last page is 0x7F
    last = inp.block_table[1, 0].item()
    assert np.all(inp.kv_cache[last, 5:].numpy() == 0x7F)


def test_sparse_single_index_and_all_skipped():
    # a list that names one row (the rest -1) returns that row and its own score;
    # a list of only -1 sees no key: zeros and -inf
    inp = syn.sparse_inputs(61, 2, num_tokens=4096, topk=64)
    idx = np.full((2, 64), -1, dtype=np.int32)
    idx[0, 37] = 1234
    out, lse = oracle.sparse_mla_decode(inp.q, inp.kv_cache, idx, inp.kv_scale, inp.softmax_scale)
    row = oracle.e4m3_decode(inp.kv_cache.numpy()[1234]) * inp.kv_scale
    q = inp.q.float().numpy().astype(np.float64)
    for h in range(q.shape[1]):
        assert np.array_equal(out[0, h], row)
        assert abs(lse[0, h] - math.fsum(q[0, h] * row) * inp.softmax_scale) < 1e-12
    assert np.all(out[1] == 0) and np.all(lse[1] == -np.inf)


def test_two_shard_merge_by_hand():
    # shard A: m = 1, l = 2, acc = [2, 4]; shard B: m = 3, l = 1, acc = [1, 0]
    # M = 3, L = 2 e^-2 + 1, out = (e^-2 [2, 4] + [1, 0]) / L, lse = 3 + ln L
    out, lse = oracle.merge_partials([(1.0, 2.0, np.array([2.0, 4.0])), (3.0, 1.0, np.array([1.0, 0.0])),
                                      (-math.inf, 0.0, np.zeros(2))])
    big_l = 2.0 * math.exp(-2.0) + 1.0
    assert np.allclose(out, [(2.0 * math.exp(-2.0) + 1.0) / big_l, 4.0 * math.exp(-2.0) / big_l], rtol=1e-15)
    assert abs(lse - (3.0 + math.log(big_l))) < 1e-15
    # a split of explicit scores agrees with the softmax written out
    s = np.array([0.5, -1.0, 2.0, 0.0])
    v = np.array([[1.0, 0.0], [0.0, 1.0], [2.0, 2.0], [-1.0, 3.0]])
    direct = oracle.softmax_attention(s, v)
    merged = oracle.merge_partials([oracle.partial_attention(s[:1], v[:1]), oracle.partial_attention(s[1:], v[1:])])
    w = np.exp(s) / np.exp(s).sum()
    assert np.allclose(direct[0], w @ v, rtol=1e-14) and np.allclose(merged[0], w @ v, rtol=1e-14)
    assert abs(merged[1] - math.log(np.exp(s).sum())) < 1e-14
