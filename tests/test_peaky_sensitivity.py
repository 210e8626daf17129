"""The peaky test case can tell a P scale of 128 from a P scale of 1 (CPU only).

aiter "Support fp8 KV caches and fp8 dots in sparse_mla_fwd on gfx942",
Accuracy and the review asking for a focused case: with one key scoring 9
above 2047 others that carry a fifth of the output, quantising p to E4M3
without the x128 scale flushes the tail (p ~ 1e-4 is below E4M3's smallest
subnormal 2^-9) and the error is large; with the scale it is small.  The
quantisation here is a model of the kernel's P step (torch's E4M3 cast),
compared with the fp64 oracle; the planted mistake (scale 1) lives only in
this CPU model.
"""

import numpy as np
import torch

import oracle
from oracle.attention import e4m3_decode
from paged_decode_attention_fp8_gb300 import synthetic as syn


def _quantised_p_attention(inp, p_scale):
    q = inp.q.double().numpy()
    cache = inp.kv_cache.numpy()
    idx = inp.topk_idx.numpy()
    outs = []
    for t in range(q.shape[0]):
        keys = e4m3_decode(cache[idx[t]]) * inp.kv_scale
        s = q[t] @ keys.T * inp.softmax_scale
        p = np.exp(s - s.max(axis=1, keepdims=True))
        pq = torch.from_numpy((p * p_scale).astype(np.float32)).to(torch.float8_e4m3fn).double().numpy()
        outs.append((pq @ keys) / (p.sum(axis=1, keepdims=True) * p_scale))
    return np.stack(outs)


def test_unscaled_p_loses_the_tail_scaled_keeps_it():
    inp = syn.sparse_peaky_inputs(4, s_q=2, num_tokens=8192)
    ref, _ = oracle.sparse_mla_decode(inp.q, inp.kv_cache, inp.topk_idx, inp.kv_scale, inp.softmax_scale)

    def rel(x):
        return np.linalg.norm((x - ref)[..., 256:]) / np.linalg.norm(ref[..., 256:])

    err_scaled = rel(_quantised_p_attention(inp, 128.0))
    err_unscaled = rel(_quantised_p_attention(inp, 1.0))
    assert err_scaled < 0.03
    assert err_unscaled > 0.15


def _dense_quantised_p_attention(inp, p_scale):
    """The dense MLA analogue: one softmax over a sequence's whole cache,
    p quantised as E4M3(p_scale * p), V = the first 512 dims of each key."""
    q = inp.q.double().numpy()[:, 0]  # s_q = 1
    cache = inp.kv_cache.numpy()
    bt = inp.block_table.numpy()
    outs = []
    for i, s_k in enumerate(inp.seqlens.numpy()):
        pages = bt[i, : (s_k + 63) // 64]
        keys = (e4m3_decode(cache[pages]) * inp.kv_scale).reshape(-1, 576)[:s_k]
        s = q[i] @ keys.T * inp.softmax_scale
        p = np.exp(s - s.max(axis=1, keepdims=True))
        pq = torch.from_numpy((p * p_scale).astype(np.float32)).to(torch.float8_e4m3fn).double().numpy()
        outs.append((pq @ keys[:, :512]) / (p.sum(axis=1, keepdims=True) * p_scale))
    return np.stack(outs)[:, None]


def test_dense_peaky_case_closed_form_and_p_scale():
    # the dense construction reproduces the page's numbers: the peak key's
    # weight 1 / (1 + 2047 e^-9) and lse = 9 + ln(1 + 2047 e^-9)
    inp = syn.mla_peaky_inputs(5, b=2, h_q=8)
    ref, lse = oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens, inp.kv_scale,
                                 inp.softmax_scale, False)
    assert np.allclose(lse, 9.0 + np.log1p(2047 * np.exp(-9.0)), atol=1e-5)

    def rel(x):
        return np.linalg.norm((x - ref)[..., 256:]) / np.linalg.norm(ref[..., 256:])

    # E4M3(64 p) keeps the tail (the dense kernel's P scale), E4M3(p) flushes it
    assert rel(_dense_quantised_p_attention(inp, 64.0)) < 0.03
    assert rel(_dense_quantised_p_attention(inp, 1.0)) > 0.15
