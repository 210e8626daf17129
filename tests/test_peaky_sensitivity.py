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
