"""The C-ABI library loads without a GPU, exports every function declared in
include/*.h, and refuses bad arguments on the host before launching anything
(no compute call is made here)."""

import ctypes
import glob
import os
import re

import pytest

import paged_decode_attention_fp8_gb300 as fm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"FP8MLA_API\s+[\w\s\*]+?\b(\w+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_symbol():
    lib = fm.lib()
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    assert names == set(fm.EXPORTED_SYMBOLS)


def test_exported_symbols_are_only_the_c_abi():
    out = os.popen(f"nm -D --defined-only {fm.LIB_PATH}").read()
    text_syms = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert text_syms == declared_functions()


def test_status_strings_and_units():
    lib = fm.lib()
    assert lib.fp8mla_status_string(0) == b"ok"
    assert b"E4M3" in lib.fp8mla_status_string(2)
    assert lib.fp8mla_metadata_units(148) == 74
    assert lib.fp8mla_metadata_units(152) == 76
    assert lib.fp8mla_metadata_units(1) == 1


def test_workspace_sizes_grow_with_batch():
    lib = fm.lib()
    a = lib.fp8mla_workspace_bytes(64, 2, 64, 76)
    b = lib.fp8mla_workspace_bytes(128, 2, 64, 76)
    # at least the bf16 partial O of every slot (b + units of them) and the quantised Q
    assert b > a > 140 * 128 * 512 * 2 + 64 * 88064
    assert a % 256 == 0


def _decode(**over):
    args = dict(q=1 << 20, kv=1 << 20, kv_dtype=fm.KV_E4M3, num_pages=16, bt=1 << 20, max_pages=8, sl=1 << 20,
                scale=1 << 20, softmax_scale=0.04, causal=1, ts=1 << 20, ns=1 << 20, units=76, ws=1 << 20,
                ws_bytes=1 << 40, out=1 << 20, lse=1 << 20, dot=fm.DOT_FP8, b=2, s_q=2, h_q=64)
    args.update(over)
    a = args
    return fm.lib().fp8mla_decode(a["q"], a["kv"], a["kv_dtype"], a["num_pages"], a["bt"], a["max_pages"], a["sl"],
                                  a["scale"], a["softmax_scale"], a["causal"], a["ts"], a["ns"], a["units"], a["ws"],
                                  a["ws_bytes"], a["out"], a["lse"], a["dot"], a["b"], a["s_q"], a["h_q"], None)


@pytest.mark.parametrize("code", [fm.KV_E4M3FNUZ, fm.KV_E5M2, fm.KV_OTHER])
def test_foreign_encodings_refused(code):
    assert _decode(kv_dtype=code) == 2


def test_missing_scale_refused():
    # an FP8 cache without its scale fails loudly (InfiniCore page: "Bad Parameter")
    assert _decode(scale=None) == 1


@pytest.mark.parametrize("over", [dict(h_q=128), dict(s_q=0), dict(q=None), dict(out=None), dict(units=0),
                                  dict(dot=7), dict(softmax_scale=0.0), dict(q=(1 << 20) + 2),
                                  dict(num_pages=0)])
def test_bad_arguments_refused(over):
    assert _decode(**over) == 1


def _decode_ext(**over):
    a = dict(q=1 << 20, kv=1 << 20, kv_dtype=fm.KV_E4M3, num_pages=16, bt=1 << 20, max_pages=8, sl=1 << 20,
             scale=None, rows=1 << 20, softmax_scale=0.04, causal=1, ts=1 << 20, ns=1 << 20, units=76, ws=1 << 20,
             ws_bytes=1 << 40, out=1 << 20, lse=1 << 20, dot=fm.DOT_FP8, b=2, s_q=2, h_q=64)
    a.update(over)
    return fm.lib().fp8mla_decode_ext(a["q"], a["kv"], a["kv_dtype"], a["num_pages"], a["bt"], a["max_pages"],
                                      a["sl"], a["scale"], a["rows"], a["softmax_scale"], a["causal"], a["ts"],
                                      a["ns"], a["units"], a["ws"], a["ws_bytes"], a["out"], a["lse"], a["dot"],
                                      a["b"], a["s_q"], a["h_q"], None)


@pytest.mark.parametrize("over", [dict(rows=None), dict(dot=fm.DOT_16BIT), dict(rows=(1 << 20) + 4),
                                  dict(h_q=128), dict(q=None)])
def test_decode_ext_refusals(over):
    # neither scale given; per-row scales with 16-bit dots; rows not 16-byte aligned; bad shapes
    assert _decode_ext(**over) == 1


def test_decode_ext_foreign_encoding_workspace_and_empty_batch():
    assert _decode_ext(kv_dtype=fm.KV_E5M2) == 2
    assert _decode_ext(ws_bytes=1024) == 3
    assert _decode_ext(b=0, q=None, out=None, lse=None) == 0


def test_small_workspace_refused():
    assert _decode(ws_bytes=1024) == 3


def test_metadata_argument_checks():
    lib = fm.lib()
    # force_splits * b > units
    assert lib.fp8mla_get_metadata(1 << 20, 64, 64, 2, 76, 2, 1 << 20, 1 << 20, None) == 1
    assert lib.fp8mla_get_metadata(1 << 20, 4, 128, 2, 76, 0, 1 << 20, 1 << 20, None) == 1
    assert lib.fp8mla_get_metadata(None, 4, 64, 2, 76, 0, 1 << 20, 1 << 20, None) == 1


def test_sparse_and_gqa_refuse_foreign_encodings_and_missing_scales():
    lib = fm.lib()
    assert lib.sparse_mla_decode(1 << 20, 1 << 20, fm.KV_E5M2, 1024, 1 << 20, 2048, 1 << 20, 0.04, 0, 1 << 20,
                                 1 << 40, 1 << 20, 1 << 20, fm.DOT_FP8, 2, 16, None) == 2
    assert lib.sparse_mla_decode(1 << 20, 1 << 20, fm.KV_E4M3, 1024, 1 << 20, 2048, None, 0.04, 0, 1 << 20,
                                 1 << 40, 1 << 20, 1 << 20, fm.DOT_FP8, 2, 16, None) == 1
    assert lib.paged_gqa_decode(1 << 20, 1 << 20, 1 << 20, fm.KV_E4M3FNUZ, 64, 1 << 20, 1 << 20, 1 << 20, 8,
                                1 << 20, 0.08, 0, 1 << 20, 1 << 40, 1 << 20, 1 << 20, 1, 32, 8, 128, 16, None) == 2
    assert lib.paged_gqa_decode(1 << 20, 1 << 20, 1 << 20, fm.KV_E4M3, 64, None, 1 << 20, 1 << 20, 8,
                                1 << 20, 0.08, 0, 1 << 20, 1 << 40, 1 << 20, 1 << 20, 1, 32, 8, 128, 16, None) == 1


def test_python_dtype_mapping():
    import torch
    assert fm.kv_dtype_code(torch.empty(1, dtype=torch.float8_e4m3fn)) == fm.KV_E4M3
    assert fm.kv_dtype_code(torch.empty(1, dtype=torch.uint8)) == fm.KV_E4M3
    assert fm.kv_dtype_code(torch.empty(1, dtype=torch.float8_e5m2)) == fm.KV_E5M2
    assert fm.kv_dtype_code(torch.empty(1, dtype=torch.int8)) == fm.KV_OTHER
    assert fm.kv_dtype_code(torch.empty(1, dtype=torch.bool)) == fm.KV_OTHER


def _cache_write(**over):
    a = dict(x=1 << 20, stride=1024, slots=1 << 20, n=4, h_kv=8, hd=128, page=16, blocks=64, dtype=fm.KV_E4M3,
             cache=1 << 20, tscale=None, rscales=1 << 20)
    a.update(over)
    return fm.lib().fp8_paged_cache_write(a["x"], a["stride"], a["slots"], a["n"], a["h_kv"], a["hd"], a["page"],
                                          a["blocks"], a["dtype"], a["cache"], a["tscale"], a["rscales"], None)


@pytest.mark.parametrize("over", [dict(tscale=1 << 20), dict(rscales=None), dict(hd=12), dict(hd=0), dict(hd=1032),
                                  dict(stride=1000), dict(stride=1020), dict(x=None), dict(slots=None),
                                  dict(cache=None), dict(x=(1 << 20) + 8), dict(cache=(1 << 20) + 4),
                                  dict(page=0), dict(blocks=0), dict(h_kv=0), dict(n=-1)])
def test_cache_write_bad_arguments_refused(over):
    assert _cache_write(**over) == 1


def test_cache_write_refuses_foreign_encodings_and_empty_is_a_no_op():
    assert _cache_write(dtype=fm.KV_E5M2) == 2
    assert _cache_write(dtype=fm.KV_E4M3FNUZ) == 2
    # nothing to write: accepted without touching the device (null pointers allowed)
    assert _cache_write(n=0, x=None, slots=None, cache=None) == 0



def _gqa(**over):
    a = dict(q=1 << 20, k=1 << 20, v=1 << 20, dtype=fm.KV_E4M3, nb=64, ks=1 << 20, vs=1 << 20, bt=1 << 20, mb=8,
             sl=1 << 20, scale=0.08, splits=1, ws=1 << 20, ws_bytes=1 << 40, out=1 << 20, lse=1 << 20, bs=2,
             h_q=32, h_kv=8, hd=128, page=16)
    a.update(over)
    return fm.lib().paged_gqa_decode(a["q"], a["k"], a["v"], a["dtype"], a["nb"], a["ks"], a["vs"], a["bt"], a["mb"],
                                     a["sl"], a["scale"], a["splits"], a["ws"], a["ws_bytes"], a["out"], a["lse"],
                                     a["bs"], a["h_q"], a["h_kv"], a["hd"], a["page"], None)


@pytest.mark.parametrize("over", [dict(hd=64), dict(page=32), dict(h_q=30), dict(h_q=136), dict(splits=-1),
                                  dict(scale=0.0), dict(nb=0), dict(mb=0), dict(q=None), dict(lse=None),
                                  dict(k=(1 << 20) + 8), dict(splits=4, ws=None), dict(splits=4, ws=(1 << 20) + 64)])
def test_gqa_shape_and_argument_refusals(over):
    assert _gqa(**over) == 1


def test_gqa_small_workspace_and_empty_batch():
    assert _gqa(splits=4, ws_bytes=256) == 3
    assert _gqa(bs=0, q=None, out=None, lse=None) == 0      # nothing to do, nothing touched


def _gqa_ext(**over):
    a = dict(q=1 << 20, k=1 << 20, v=1 << 20, dtype=fm.KV_E4M3, nb=64, ks=1 << 20, vs=1 << 20, rows=0,
             bt=1 << 20, mb=8, sl=1 << 20, scale=0.08, q_len=1, mask=None, window=0, sinks=None, splits=1,
             ws=1 << 20, ws_bytes=1 << 40, out=1 << 20, lse=1 << 20, bs=2, h_q=32, h_kv=8, hd=128, page=16)
    a.update(over)
    return fm.lib().paged_gqa_decode_ext(a["q"], a["k"], a["v"], a["dtype"], a["nb"], a["ks"], a["vs"], a["rows"],
                                         a["bt"], a["mb"], a["sl"], a["scale"], a["q_len"], a["mask"], a["window"],
                                         a["sinks"], a["splits"], a["ws"], a["ws_bytes"], a["out"], a["lse"],
                                         a["bs"], a["h_q"], a["h_kv"], a["hd"], a["page"], None)


@pytest.mark.parametrize("over", [dict(q_len=0), dict(q_len=5), dict(q_len=2, h_q=72, h_kv=8), dict(window=-1),
                                  dict(rows=1, ks=(1 << 20) + 4), dict(rows=1, vs=(1 << 20) + 8), dict(ks=None),
                                  dict(hd=64), dict(h_q=30)])
def test_gqa_ext_argument_refusals(over):
    # group 4: q_len * group must stay <= 16; per-row scale arrays must be 16-byte aligned
    assert _gqa_ext(**over) == 1


def test_gqa_ext_foreign_encoding_and_empty_batch():
    assert _gqa_ext(dtype=fm.KV_E4M3FNUZ) == 2
    assert _gqa_ext(bs=0, q=None, out=None, lse=None, q_len=4) == 0


def _sparse(**over):
    a = dict(q=1 << 20, kv=1 << 20, dtype=fm.KV_E4M3, n=131072, idx=1 << 20, topk=2048, scale=1 << 20, sm=0.04,
             splits=1, ws=1 << 20, ws_bytes=1 << 40, out=1 << 20, lse=1 << 20, dot=fm.DOT_FP8, s_q=2, h_q=16)
    a.update(over)
    return fm.lib().sparse_mla_decode(a["q"], a["kv"], a["dtype"], a["n"], a["idx"], a["topk"], a["scale"], a["sm"],
                                      a["splits"], a["ws"], a["ws_bytes"], a["out"], a["lse"], a["dot"], a["s_q"],
                                      a["h_q"], None)


@pytest.mark.parametrize("over", [dict(h_q=17), dict(topk=0), dict(dot=fm.DOT_16BIT), dict(n=0), dict(sm=0.0),
                                  dict(splits=-1), dict(q=None), dict(idx=None), dict(out=(1 << 20) + 4),
                                  dict(n=1 << 31), dict(splits=4, ws=None)])
def test_sparse_argument_refusals(over):
    assert _sparse(**over) == 1


def test_sparse_small_workspace_and_no_tokens():
    assert _sparse(splits=4, ws_bytes=256) == 3
    assert _sparse(s_q=0, q=None, out=None, lse=None) == 0


def _no_alloc(**over):
    a = dict(q=1 << 20, kv=1 << 20, dtype=fm.KV_E4M3, np_=16, bt=1 << 20, mp=8, sl=1 << 20, scale=1 << 20, sm=0.04,
             causal=1, out=1 << 20, lse=1 << 20, dot=fm.DOT_FP8, b=2, s_q=2, h_q=64)
    a.update(over)
    return fm.lib().fp8mla_decode_no_alloc(a["q"], a["kv"], a["dtype"], a["np_"], a["bt"], a["mp"], a["sl"],
                                           a["scale"], a["sm"], a["causal"], a["out"], a["lse"], a["dot"], a["b"],
                                           a["s_q"], a["h_q"], None)


def test_no_alloc_host_checks():
    assert _no_alloc(b=65) == 3                 # beyond the fixed array: refused before any launch
    assert _no_alloc(dtype=fm.KV_E5M2) == 2
    assert _no_alloc(h_q=128) == 1              # s_q * h_q > 128
    assert _no_alloc(b=0, q=None, out=None, lse=None) == 0


def test_gqa_split_rule_on_the_host():
    lib = fm.lib()
    # forced: capped at the 128-token steps the longest context has
    assert lib.paged_gqa_num_splits(1, 8, 16384, 152, 4) == 4
    assert lib.paged_gqa_num_splits(1, 8, 256, 152, 8) == 2
    # a grid that fills the GPU (32 x 8 = 256 CTAs >= 0.8 x 152): about six CTAs per SM,
    # ceil(6 * 152 / 256) = 4 pieces, each at least 8 steps (16384 / 128 / 8 = 16 allows it)
    assert lib.paged_gqa_num_splits(32, 8, 16384, 152, 0) == 4
    assert lib.paged_gqa_num_splits(256, 8, 1024, 152, 0) == 1     # 8 steps: pieces would be shorter
    # a small grid: the fewest pieces whose wave efficiency is within 85 % of the best up to 16;
    # 8 CTAs x s pieces fit in one wave of 152 for s <= 16, efficiency 8 s / 152, best at 16,
    # and 8 s / 152 >= 0.85 * 128 / 152 first at s = 14
    assert lib.paged_gqa_num_splits(1, 8, 16384, 152, 0) == 14
    assert lib.paged_gqa_num_splits(1, 8, 128, 152, 0) == 1        # one step: nothing to split
    # the extended entry with a window: nearly equal pieces need no balancing, so a grid that
    # fills the GPU (256 CTAs) is not split; a small grid still splits to fill its wave
    assert lib.paged_gqa_ext_num_splits(32, 8, 16384, 4, 4096, 152, 0) == 1
    assert lib.paged_gqa_ext_num_splits(32, 8, 16384, 4, 0, 152, 0) == 4   # no window: the plain rule
    assert lib.paged_gqa_ext_num_splits(1, 8, 16384, 4, 4096, 152, 0) == 14  # a small grid: waves
    assert lib.paged_gqa_ext_num_splits(32, 8, 16384, 4, 4096, 152, 3) == 3  # forced
