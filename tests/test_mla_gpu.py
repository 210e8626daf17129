"""Dense MLA decode on the GPU against the fp64 oracle (through the C ABI).

Workloads follow the FlashMLA "update fp8 support" page: the tiny case
(b=2, s_q=1, h_q=16, cache {256, 300}), the MTP decode shape (b=64, s_q=2,
h_q=64, s_k uniform in [2048, 6144]) and the fixed long cache (s_k=8196).
"""

import math

import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_fp8_gb300 as fm
from paged_decode_attention_fp8_gb300 import synthetic as syn
from tests.parity import assert_close, compare, record

pytestmark = pytest.mark.gpu

MODES = ["fp8", "bf16"]


def to_dev(inp):
    dev = torch.device("cuda")
    return dict(q=inp.q.to(dev), kv=inp.kv_cache.to(dev), bt=inp.block_table.to(dev),
                sl=inp.seqlens.to(dev),
                scale=torch.tensor([inp.kv_scale], dtype=torch.float32, device=dev))


def run_mla(inp, mode, force_splits=0, units=None, d=None):
    d = d or to_dev(inp)
    ts, ns = fm.get_metadata(d["sl"], inp.h_q, inp.s_q, num_units=units, force_splits=force_splits)
    out, lse = fm.decode(d["q"], d["kv"], d["bt"], d["sl"], d["scale"], inp.softmax_scale, inp.causal,
                         ts, ns, dot_mode=mode)
    torch.cuda.synchronize()
    return out, lse


def ref(inp, batches=None):
    return oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens, inp.kv_scale,
                             inp.softmax_scale, inp.causal, batches=batches)


def check(inp, mode, force_splits=0, units=None, name=None):
    out, lse = run_mla(inp, mode, force_splits, units)
    ro, rl = ref(inp)
    m = compare(out, lse, ro, rl, mode)
    if name:
        record(name, m)
    assert_close(m, mode)
    assert fm.last_device_error() == 0
    return m


# ------------------------------------------------------------ metadata ----


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("force", [0, 1, 2, 3])
def test_metadata_bit_exact(seed, force):
    rng = np.random.default_rng(seed)
    b = int(rng.integers(1, 40))
    seqlens = rng.integers(0, 5000, size=b).astype(np.int32)
    seqlens[rng.random(b) < 0.15] = 0
    units = fm.metadata_units()
    if force * b > units:
        force = 0
    sl = torch.from_numpy(seqlens).cuda()
    ts, ns = fm.get_metadata(sl, 16, 1, num_units=units, force_splits=force)
    exp_ts, exp_ns = oracle.schedule(seqlens, units, force_splits=force)
    assert np.array_equal(ts.cpu().numpy(), exp_ts)
    assert np.array_equal(ns.cpu().numpy(), exp_ns)


def test_metadata_headline_bit_exact():
    seqlens = np.array(syn.uniform_seqlens(2, 64, 2048, 6144), dtype=np.int32)
    units = fm.metadata_units()
    ts, ns = fm.get_metadata(torch.from_numpy(seqlens).cuda(), 64, 2, num_units=units)
    exp_ts, exp_ns = oracle.schedule(seqlens, units)
    assert np.array_equal(ts.cpu().numpy(), exp_ts) and np.array_equal(ns.cpu().numpy(), exp_ns)


# --------------------------------------------------------- tiny config ----


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("force", [0, 1, 2, 3])
def test_tiny_config(mode, force):
    inp = syn.mla_inputs(1, 2, 1, 16, [256, 300], causal=False, spare_pages=7)
    assert inp.kv_cache.shape[0] == 16
    check(inp, mode, force_splits=force, name=f"tiny_b2_force{force}_{mode}")


@pytest.mark.parametrize("mode", MODES)
def test_ragged_lengths_and_empty_rows(mode):
    # lengths around page edges, an empty cache and a causal cut with s_k = 1 < s_q
    seqlens = [0, 1, 63, 64, 65, 127, 128, 129, 1000, 2]
    inp = syn.mla_inputs(21, len(seqlens), 2, 64, seqlens, causal=True, spare_pages=5)
    for force in (0, 2):
        check(inp, mode, force_splits=force)


@pytest.mark.parametrize("mode", MODES)
def test_padded_rows_and_non_causal(mode):
    inp = syn.mla_inputs(22, 5, 2, 24, [700, 64, 1, 130, 5000], causal=False, spare_pages=3)
    check(inp, mode)


# ------------------------------------------------------- headline shape ----


@pytest.mark.parametrize("mode", MODES)
def test_headline_mtp_decode(mode):
    seqlens = syn.uniform_seqlens(2, 64, 2048, 6144)
    inp = syn.mla_inputs(2, 64, 2, 64, seqlens, causal=True, spare_pages=64)
    check(inp, mode, name=f"headline_b64_sq2_{mode}")


@pytest.mark.parametrize("b", [32, 48, 64, 128])
def test_fixed_long_cache_sampled(b):
    # the FlashMLA page's H20 table: cache 8196, MTP = 2, 64 heads, FP8 dots;
    # the whole batch runs, four sequences spread over it are checked
    inp = syn.mla_inputs(3, b, 2, 64, [8196] * b, causal=True, value_pages=512)
    out, lse = run_mla(inp, "fp8")
    picks = [0, b // 3, (2 * b) // 3, b - 1]
    ro, rl = ref(inp, batches=picks)
    m = compare(out[picks], lse[picks], ro[picks], rl[picks], "fp8")
    record(f"long_b{b}_sk8196_fp8_sampled", m)
    assert_close(m, "fp8")
    assert fm.last_device_error() == 0


@pytest.mark.parametrize("mode", MODES)
def test_fixed_4096_mtp_decode(mode):
    # the FlashMLA page's H800 run: b = 64, s_q = 2, every s_k = 4096, causal
    inp = syn.mla_inputs(12, 64, 2, 64, [4096] * 64, causal=True, spare_pages=16)
    check(inp, mode, name=f"fixed_b64_sq2_sk4096_{mode}")


@pytest.mark.parametrize("mode", MODES)
def test_peaky_tail_kept_with_split_off(mode):
    # one key +9 above 2047 that carry a fifth of the output (aiter page,
    # Accuracy), on the dense kernel: its P scale (E4M3(64 p) with FP8 dots)
    # must keep the tail, which an unscaled E4M3 P would flush
    inp = syn.mla_peaky_inputs(13, b=2, h_q=64, s_k=2048)
    out, lse = run_mla(inp, mode, force_splits=1)
    ro, rl = ref(inp)
    m = compare(out, lse, ro, rl, mode)
    record(f"dense_peaky_splits1_{mode}", m)
    assert_close(m, mode)
    mv = compare(out[..., 256:], lse, ro[..., 256:], rl, mode)
    record(f"dense_peaky_value_dims_{mode}", mv)
    assert mv["rel_l2"] < (5e-2 if mode == "fp8" else 1e-2)
    assert fm.last_device_error() == 0


# --------------------------------------------------------- invariances ----


def test_page_relabelling_bit_identical():
    seqlens = [300, 1, 64, 777, 2048]
    inp = syn.mla_inputs(5, 5, 2, 64, seqlens, causal=True, spare_pages=20)
    out_a, lse_a = run_mla(inp, "fp8")
    perm = np.random.default_rng(9).permutation(inp.kv_cache.shape[0])
    cache = np.empty_like(inp.kv_cache.numpy())
    cache[perm] = inp.kv_cache.numpy()
    moved = syn.MLAInputs(q=inp.q, kv_cache=torch.from_numpy(cache),
                          block_table=torch.from_numpy(perm[inp.block_table.numpy()].astype(np.int32)),
                          seqlens=inp.seqlens, kv_scale=inp.kv_scale, softmax_scale=inp.softmax_scale,
                          causal=True)
    out_b, lse_b = run_mla(moved, "fp8")
    assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)


def test_run_to_run_bit_identical():
    seqlens = syn.uniform_seqlens(4, 16, 100, 3000)
    inp = syn.mla_inputs(4, 16, 2, 64, seqlens, causal=True)
    d = to_dev(inp)
    a = run_mla(inp, "fp8", d=d)
    b = run_mla(inp, "fp8", d=d)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("mode", MODES)
def test_forced_split_counts_stay_within_tolerance(mode):
    # each split has its own running max, so FP8 P is quantised on a different
    # grid per split: every split count must meet the oracle tolerance, and
    # with 16-bit dots the split counts must also agree closely with each other
    seqlens = [1500, 2100, 900]
    inp = syn.mla_inputs(6, 3, 2, 64, seqlens, causal=True)
    ro, rl = ref(inp)
    base = None
    for k in (1, 2, 5, 8):
        o, l = run_mla(inp, mode, force_splits=k)
        m = compare(o, l, ro, rl, mode)
        record(f"forced_splits_{k}_{mode}", m)
        assert_close(m, mode)
        if base is None:
            base = (o, l)
        elif mode == "bf16":
            rel = (o.float() - base[0].float()).norm() / base[0].float().norm()
            assert rel < 5e-3 and (l - base[1]).abs().max() < 1e-3


def test_poisoned_tail_does_not_leak():
    # every slot past a sequence end and every spare page holds 0x7F (NaN)
    inp = syn.mla_inputs(7, 3, 2, 64, [65, 100, 191], causal=True, spare_pages=8)
    out, lse = run_mla(inp, "fp8")
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_bad_page_index_is_reported_not_faulted():
    inp = syn.mla_inputs(8, 2, 1, 16, [100, 100], causal=False)
    inp.block_table[1, 1] = inp.kv_cache.shape[0] + 5
    run_mla(inp, "fp8")
    assert fm.last_device_error() & fm.DEV_BAD_PAGE
    assert fm.last_device_error() == 0   # read-and-clear


@pytest.mark.parametrize("mode", MODES)
def test_q_written_just_before_the_call_is_seen(mode):
    # Q is produced by a torch kernel on the same stream right before the
    # call (as a projection GEMM would leave it): the call's first kernel
    # must wait for that write before it reads Q, and the decode kernel
    # (which reads the bf16 Q again for 16-bit dots) after it
    inp = syn.mla_inputs(14, 8, 2, 64, syn.uniform_seqlens(14, 8, 100, 3000), causal=True)
    d = to_dev(inp)
    src = d["q"].clone()
    ts, ns = fm.get_metadata(d["sl"], inp.h_q, inp.s_q)
    ro, rl = ref(inp)
    for _ in range(3):
        q = torch.zeros_like(src)
        torch.cuda.synchronize()
        q.add_(src * 1.0)  # two torch kernels, enqueued just ahead of the decode
        out, lse = fm.decode(q, d["kv"], d["bt"], d["sl"], d["scale"], inp.softmax_scale, True, ts, ns,
                             dot_mode=mode)
        torch.cuda.synchronize()
        assert_close(compare(out, lse, ro, rl, mode), mode)
