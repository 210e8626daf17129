"""Pins of the oracle's XQA options for paged GQA decode (FlashInfer "add xqa
fp8 mha and fp8 kv cache": speculative-decoding block with a mask, sliding
window, attention sinks) against facts that do not come from that code:

* special cases that reduce to the plain decode: one query token with every
  option off, the default mask = an explicit lower-triangular mask, a window
  at least the cache length, a sink of -inf;
* closed forms: a one-key window returns the query's own value and score; a
  sink s gives lse' = logaddexp(lse, s) and out' = out * e^(lse - lse');
* the masked-row rule of the same page: a row that sees no key gives zeros
  (and lse = the sink, or -inf), never the mean of V;
* the causal block agrees with the dense MLA oracle's causal alignment;
* brute force with its own visibility test, correctly rounded sums and the
  E4M3 table.
"""

import math

import numpy as np

import oracle
from oracle.attention import e4m3_decode, gqa_decode_ext, mla_visible_keys, spec_visible
from paged_decode_attention_fp8_gb300 import synthetic as syn

H_Q, H_KV, HD = 4, 2, 16


def _inputs(seed, seqlens, q_len):
    inp = syn.gqa_inputs(seed, len(seqlens), seqlens, h_q=H_Q, h_kv=H_KV, hd=HD, spare_blocks=2)
    q = syn.to_bf16(syn.normal(seed, 50, (len(seqlens), q_len, H_Q, HD)))
    return inp, q


def _run(inp, q, **kw):
    return gqa_decode_ext(q, inp.k_cache, inp.v_cache, inp.block_table, inp.seqlens, inp.k_scale, inp.v_scale,
                          inp.softmax_scale, **kw)


def test_single_query_equals_plain_decode():
    inp, q = _inputs(51, [40, 3, 17], 1)
    a = _run(inp, q)
    b = oracle.gqa_decode(q[:, 0], inp.k_cache, inp.v_cache, inp.block_table, inp.seqlens, inp.k_scale,
                          inp.v_scale, inp.softmax_scale)
    assert np.array_equal(a[0][:, 0], b[0]) and np.array_equal(a[1][:, 0], b[1])


def test_default_mask_is_causal_and_matches_mla_alignment():
    inp, q = _inputs(52, [40, 9], 3)
    tri = np.broadcast_to(np.tril(np.ones((3, 3), dtype=bool)), (2, 3, 3))
    a = _run(inp, q)
    b = _run(inp, q, spec_mask=tri)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    for s_k in (3, 9, 40):
        for i in range(3):
            assert spec_visible(s_k, 3, i).sum() == mla_visible_keys(s_k, 3, i, True)


def test_window_closed_forms():
    inp, q = _inputs(53, [40, 9], 2)
    a = _run(inp, q)
    assert all(np.array_equal(x, y) for x, y in zip(a, _run(inp, q, window=40)))
    out, lse = _run(inp, q, window=1)
    kc, vc = inp.k_cache.numpy(), inp.v_cache.numpy()
    bt = inp.block_table.numpy()
    qf = q.float().numpy().astype(np.float64)
    for b, s_k in enumerate(inp.seqlens.tolist()):
        for i in range(2):
            p = s_k - 2 + i
            blk, off = int(bt[b, p // 16]), p % 16
            for h in range(H_Q):
                kvh = h // (H_Q // H_KV)
                k = e4m3_decode(kc[blk, kvh, off]) * inp.k_scale
                v = e4m3_decode(vc[blk, kvh, off]) * inp.v_scale
                assert np.allclose(out[b, i, h], v, rtol=0, atol=0)
                assert abs(lse[b, i, h] - (k @ qf[b, i, h]) * inp.softmax_scale) < 1e-12


def test_sink_closed_form():
    inp, q = _inputs(54, [40, 9], 2)
    out, lse = _run(inp, q)
    sinks = np.array([0.5, -3.0, 2.0, 7.5])
    out_s, lse_s = _run(inp, q, sinks=sinks)
    want_lse = np.logaddexp(lse, sinks[None, None, :])
    assert np.allclose(lse_s, want_lse, rtol=0, atol=1e-12)
    assert np.allclose(out_s, out * np.exp(lse - want_lse)[..., None], rtol=1e-12, atol=1e-15)
    none = _run(inp, q, sinks=np.full(H_Q, -np.inf))
    assert np.array_equal(none[0], out) and np.array_equal(none[1], lse)


def test_fully_masked_rows_give_zeros():
    inp, q = _inputs(55, [40, 9], 2)
    mask = np.ones((2, 2, 2), dtype=bool)
    mask[:, 1, :] = False                   # token 1 sees nothing of the block ...
    out, lse = _run(inp, q, spec_mask=mask, window=1)   # ... and the window leaves only itself
    assert np.all(out[:, 1] == 0) and np.all(lse[:, 1] == -np.inf)
    assert np.all(np.isfinite(lse[:, 0]))
    out_s, lse_s = _run(inp, q, spec_mask=mask, window=1, sinks=np.array([1.0, 2.0, 3.0, 4.0]))
    assert np.all(out_s[:, 1] == 0) and np.array_equal(lse_s[:, 1], np.broadcast_to([1.0, 2.0, 3.0, 4.0], (2, 4)))


def test_brute_force():
    seqlens, q_len, window = [23, 5], 3, 6
    inp, q = _inputs(56, seqlens, q_len)
    mask = syn.uniform(56, 51, 2 * q_len * q_len).reshape(2, q_len, q_len) > 0.4
    sinks = np.array([0.0, -1.0, 1.5, -np.inf])
    out, lse = _run(inp, q, spec_mask=mask, window=window, sinks=sinks)
    kc, vc = inp.k_cache.numpy(), inp.v_cache.numpy()
    bt = inp.block_table.numpy()
    qf = q.float().numpy().astype(np.float64)
    for b, s_k in enumerate(seqlens):
        for i in range(q_len):
            pos = s_k - q_len + i
            for h in range(H_Q):
                kvh = h // (H_Q // H_KV)
                terms, vals = [], []
                for j in range(s_k):
                    if pos - j >= window:
                        continue
                    if j >= s_k - q_len and not mask[b, i, j - (s_k - q_len)]:
                        continue
                    blk, off = int(bt[b, j // 16]), j % 16
                    k = [float(e4m3_decode(c)) * inp.k_scale for c in kc[blk, kvh, off]]
                    terms.append(math.fsum(qf[b, i, h, c] * k[c] for c in range(HD)) * inp.softmax_scale)
                    vals.append([float(e4m3_decode(c)) * inp.v_scale for c in vc[blk, kvh, off]])
                logits = terms + ([sinks[h]] if sinks[h] != -np.inf else [])
                if not logits:
                    assert np.all(out[b, i, h] == 0) and lse[b, i, h] == -np.inf
                    continue
                m = max(logits)
                w = [math.exp(t - m) for t in terms]
                denom = math.fsum(w + ([math.exp(sinks[h] - m)] if sinks[h] != -np.inf else []))
                want = [math.fsum(w[j] * vals[j][c] for j in range(len(w))) / denom for c in range(HD)]
                assert np.allclose(out[b, i, h], want, rtol=1e-12, atol=1e-14)
                assert abs(lse[b, i, h] - (m + math.log(denom))) < 1e-12
