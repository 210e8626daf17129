"""FP8 (E4M3) paged decode attention for GB300 (sm_103a).

Python binding of ``libfp8mla.so`` (declared in ``include/fp8mla.h``).  This
module only marshals arguments: it checks dtypes and shapes, allocates
outputs with torch when the caller does not pass them, and hands raw device
pointers and the current CUDA stream to the C ABI.  Every step of the
attention runs in the library's CUDA kernels; there is no other code path,
and a missing library is an error.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8mla.so")

OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported KV cache encoding",
                3: "workspace too small", 4: "CUDA error", 5: "device-side error"}
DOT_16BIT = 0
DOT_FP8 = 1
KV_E4M3, KV_E4M3FNUZ, KV_E5M2, KV_OTHER = 0, 1, 2, 3

DEV_WAIT_TIMEOUT = 0x1
DEV_BAD_PAGE = 0x2
DEV_BAD_SEQLEN = 0x4
DEV_BAD_INDEX = 0x8
DEV_BAD_SLOT = 0x10

MLA_D, MLA_DV, MLA_PAGE, MLA_ROWS = 576, 512, 64, 128


class FP8MLAError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} (status {status})")
        self.status = status


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "fp8mla_metadata_units": (_I, [_I]),
    "fp8mla_get_metadata": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "fp8mla_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "fp8mla_decode": (_I, [_P, _P, _I, _I, _P, _I, _P, _P, _F, _I, _P, _P, _I, _P, _SZ, _P, _P, _I, _I, _I, _I,
                           _P]),
    "fp8mla_decode_ext": (_I, [_P, _P, _I, _I, _P, _I, _P, _P, _P, _F, _I, _P, _P, _I, _P, _SZ, _P, _P, _I, _I, _I,
                               _I, _P]),
    "sparse_mla_decode": (_I, [_P, _P, _I, ctypes.c_int64, _P, _I, _P, _F, _I, _P, _SZ, _P, _P, _I, _I, _I, _P]),
    "sparse_mla_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "paged_gqa_decode": (_I, [_P, _P, _P, _I, _I, _P, _P, _P, _I, _P, _F, _I, _P, _SZ, _P, _P, _I, _I, _I, _I, _I,
                              _P]),
    "paged_gqa_decode_ext": (_I, [_P, _P, _P, _I, _I, _P, _P, _I, _P, _I, _P, _F, _I, _P, _I, _P, _I, _P, _SZ,
                                  _P, _P, _I, _I, _I, _I, _I, _P]),
    "paged_gqa_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "paged_gqa_num_splits": (_I, [_I, _I, _I, _I, _I]),
    "paged_gqa_ext_num_splits": (_I, [_I, _I, _I, _I, _I, _I, _I]),
    "fp8mla_decode_no_alloc": (_I, [_P, _P, _I, _I, _P, _I, _P, _P, _F, _I, _P, _P, _I, _I, _I, _I, _P]),
    "fp8_paged_cache_write": (_I, [_P, ctypes.c_int64, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    "fp8mla_get_last_device_error": (_I, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "fp8mla_get_wait_timeout_site": (_I, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "fp8mla_set_wait_test": (_I, [ctypes.c_int32, ctypes.c_uint64]),
    "fp8mla_set_stage_timing": (_I, [ctypes.c_int]),
    "fp8mla_get_stage_times": (_I, [_P, ctypes.POINTER(ctypes.c_float)]),
    "fp8mla_status_string": (ctypes.c_char_p, [_I]),
}

EXPORTED_SYMBOLS = tuple(_SIGNATURES)


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m paged_decode_attention_fp8_gb300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(status: int, where: str) -> None:
    if status != OK:
        raise FP8MLAError(status, where)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def kv_dtype_code(t: torch.Tensor) -> int:
    """OCP E4M3 (typed or as raw uint8 bytes) is accepted; other encodings are named for refusal."""
    if t.dtype in (torch.float8_e4m3fn, torch.uint8):
        return KV_E4M3
    if t.dtype == getattr(torch, "float8_e4m3fnuz", None):
        return KV_E4M3FNUZ
    if t.dtype in (torch.float8_e5m2, getattr(torch, "float8_e5m2fnuz", torch.float8_e5m2)):
        return KV_E5M2
    return KV_OTHER


def _dot(mode) -> int:
    if mode in ("fp8", DOT_FP8):
        return DOT_FP8
    if mode in ("bf16", "16bit", DOT_16BIT):
        return DOT_16BIT
    raise ValueError(f"dot mode {mode!r}")


def _need(t: torch.Tensor, name: str, dtype=None, dim=None) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dims, got {t.dim()}")


def num_sms(device=None) -> int:
    return torch.cuda.get_device_properties(device or torch.cuda.current_device()).multi_processor_count


# -------------------------------------------------------------- dense MLA --


def metadata_units(sms: int | None = None) -> int:
    return lib().fp8mla_metadata_units(num_sms() if sms is None else sms)


def workspace_bytes(b: int, s_q: int, h_q: int, num_units: int) -> int:
    return lib().fp8mla_workspace_bytes(b, s_q, h_q, num_units)


def get_metadata(cache_seqlens: torch.Tensor, h_q: int, s_q: int, num_units: int | None = None,
                 force_splits: int = 0, tile_sched: torch.Tensor | None = None,
                 num_splits: torch.Tensor | None = None):
    """(tile_sched int32 [num_units, 8], num_splits int32 [b + 1]) for ``decode``."""
    _need(cache_seqlens, "cache_seqlens", torch.int32, 1)
    dev = cache_seqlens.device
    units = metadata_units() if num_units is None else num_units
    b = cache_seqlens.shape[0]
    if tile_sched is None:
        tile_sched = torch.empty((units, 8), dtype=torch.int32, device=dev)
    if num_splits is None:
        num_splits = torch.empty((b + 1,), dtype=torch.int32, device=dev)
    _check(lib().fp8mla_get_metadata(_ptr(cache_seqlens), b, h_q, s_q, units, force_splits,
                                     _ptr(tile_sched), _ptr(num_splits), _stream(dev)),
           "fp8mla_get_metadata")
    return tile_sched, num_splits


def decode(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
           cache_seqlens: torch.Tensor, kv_scale: torch.Tensor, softmax_scale: float | None = None,
           causal: bool = True, tile_sched: torch.Tensor | None = None,
           num_splits: torch.Tensor | None = None, dot_mode="fp8", out: torch.Tensor | None = None,
           lse: torch.Tensor | None = None, workspace: torch.Tensor | None = None):
    """Dense MLA decode.  q bf16 [b, s_q, h_q, 576]; kv_cache E4M3 [num_pages, 64, 576];
    kv_scale float32 [1] (per tensor) or [num_pages, 64] / [num_pages, 1, 64] (one scale per
    cached row, FP8 dots only).

    Returns (out bf16 [b, s_q, h_q, 512], lse float32 [b, s_q, h_q]).
    """
    _need(q, "q", torch.bfloat16, 4)
    _need(kv_cache, "kv_cache", None, 3)
    _need(block_table, "block_table", torch.int32, 2)
    _need(cache_seqlens, "cache_seqlens", torch.int32, 1)
    _need(kv_scale, "kv_scale", torch.float32)
    b, s_q, h_q, d = q.shape
    if d != MLA_D or tuple(kv_cache.shape[1:]) != (MLA_PAGE, MLA_D):
        raise ValueError("dense MLA needs q [..., 576] and kv_cache [num_pages, 64, 576]")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(MLA_D)
    if tile_sched is None or num_splits is None:
        tile_sched, num_splits = get_metadata(cache_seqlens, h_q, s_q)
    units = tile_sched.shape[0]
    if out is None:
        out = torch.empty((b, s_q, h_q, MLA_DV), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((b, s_q, h_q), dtype=torch.float32, device=q.device)
    need = workspace_bytes(b, s_q, h_q, units)
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=q.device)
    if kv_scale.numel() != 1:  # one scale per cached row
        if kv_scale.numel() != kv_cache.shape[0] * MLA_PAGE:
            raise ValueError("per-row kv_scale must hold num_pages * 64 floats")
        _check(lib().fp8mla_decode_ext(_ptr(q), _ptr(kv_cache), kv_dtype_code(kv_cache), kv_cache.shape[0],
                                       _ptr(block_table), block_table.shape[1], _ptr(cache_seqlens), None,
                                       _ptr(kv_scale), float(softmax_scale), 1 if causal else 0, _ptr(tile_sched),
                                       _ptr(num_splits), units, _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse),
                                       _dot(dot_mode), b, s_q, h_q, _stream(q.device)),
               "fp8mla_decode_ext")
        return out, lse
    _check(lib().fp8mla_decode(_ptr(q), _ptr(kv_cache), kv_dtype_code(kv_cache), kv_cache.shape[0],
                               _ptr(block_table), block_table.shape[1], _ptr(cache_seqlens), _ptr(kv_scale),
                               float(softmax_scale), 1 if causal else 0, _ptr(tile_sched), _ptr(num_splits),
                               units, _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _ptr(out), _ptr(lse), _dot(dot_mode), b, s_q, h_q, _stream(q.device)),
           "fp8mla_decode")
    return out, lse


NO_ALLOC_MAX_BATCH = 64


def decode_no_alloc(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                    cache_seqlens: torch.Tensor, kv_scale: torch.Tensor, softmax_scale: float | None = None,
                    causal: bool = True, dot_mode="fp8", out: torch.Tensor | None = None,
                    lse: torch.Tensor | None = None):
    """Dense MLA decode that needs no schedule or workspace from the caller.

    For callers that cannot allocate device memory: the library keeps the
    scratch in a fixed array of its own (one work unit per sequence, no
    split-KV), so only inputs and outputs are passed; b <= 64.  Calls that
    overlap on the GPU share that array and race.  Returns (out, lse) like
    ``decode`` (out / lse are allocated here only when not given).
    """
    _need(q, "q", torch.bfloat16, 4)
    _need(kv_cache, "kv_cache", None, 3)
    _need(block_table, "block_table", torch.int32, 2)
    _need(cache_seqlens, "cache_seqlens", torch.int32, 1)
    _need(kv_scale, "kv_scale", torch.float32)
    b, s_q, h_q, d = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(MLA_D)
    if out is None:
        out = torch.empty((b, s_q, h_q, MLA_DV), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((b, s_q, h_q), dtype=torch.float32, device=q.device)
    _check(lib().fp8mla_decode_no_alloc(_ptr(q), _ptr(kv_cache), kv_dtype_code(kv_cache), kv_cache.shape[0],
                                        _ptr(block_table), block_table.shape[1], _ptr(cache_seqlens),
                                        _ptr(kv_scale), float(softmax_scale), 1 if causal else 0, _ptr(out),
                                        _ptr(lse), _dot(dot_mode), b, s_q, h_q, _stream(q.device)),
           "fp8mla_decode_no_alloc")
    return out, lse


# ------------------------------------------------------------- sparse MLA --


def sparse_workspace_bytes(s_q: int, h_q: int, topk: int, num_splits: int = 0) -> int:
    return lib().sparse_mla_workspace_bytes(s_q, h_q, topk, num_splits)


def sparse_mla_decode(q: torch.Tensor, kv_cache: torch.Tensor, topk_idx: torch.Tensor,
                      kv_scale: torch.Tensor, softmax_scale: float | None = None, num_splits: int = 0,
                      dot_mode="fp8", out=None, lse=None, workspace=None):
    """Top-k sparse MLA decode.  q bf16 [s_q, h_q, 512]; kv_cache E4M3 [num_tokens, 512];
    topk_idx int32 [s_q, topk] (-1 = skip).  Returns (out bf16 [s_q, h_q, 512], lse [s_q, h_q])."""
    _need(q, "q", torch.bfloat16, 3)
    _need(kv_cache, "kv_cache", None, 2)
    _need(topk_idx, "topk_idx", torch.int32, 2)
    _need(kv_scale, "kv_scale", torch.float32)
    s_q, h_q, d = q.shape
    topk = topk_idx.shape[1]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((s_q, h_q, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((s_q, h_q), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = sparse_workspace_bytes(s_q, h_q, topk, num_splits)
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=q.device)
    _check(lib().sparse_mla_decode(_ptr(q), _ptr(kv_cache), kv_dtype_code(kv_cache), kv_cache.shape[0],
                                   _ptr(topk_idx), topk, _ptr(kv_scale), float(softmax_scale), num_splits,
                                   _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _ptr(out), _ptr(lse), _dot(dot_mode), s_q, h_q, _stream(q.device)),
           "sparse_mla_decode")
    return out, lse


# -------------------------------------------------------------------- GQA --


def gqa_num_splits(bs: int, h_kv: int, max_seqlen: int, num_splits: int = 0, sms: int | None = None) -> int:
    return lib().paged_gqa_num_splits(bs, h_kv, max_seqlen, num_sms() if sms is None else sms, num_splits)


def gqa_ext_num_splits(bs: int, h_kv: int, max_seqlen: int, q_len: int = 1, window: int = 0, num_splits: int = 0,
                       sms: int | None = None) -> int:
    """The key shards paged_gqa_decode_ext uses (window-aware; never more than gqa_num_splits)."""
    return lib().paged_gqa_ext_num_splits(bs, h_kv, max_seqlen, q_len, window, num_sms() if sms is None else sms,
                                          num_splits)


def gqa_workspace_bytes(bs: int, h_q: int, head_dim: int, max_splits: int) -> int:
    return lib().paged_gqa_workspace_bytes(bs, h_q, head_dim, max_splits)


def paged_gqa_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                     block_table: torch.Tensor, seqlens: torch.Tensor, k_scale: torch.Tensor,
                     v_scale: torch.Tensor, softmax_scale: float | None = None, num_splits: int = 0,
                     max_seqlen: int | None = None, out=None, lse=None, workspace=None):
    """Paged GQA decode.  q bf16 [bs, h_q, hd]; caches E4M3 [num_blocks, h_kv, page, hd].
    Returns (out bf16 [bs, h_q, hd], lse [bs, h_q])."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", None, 4)
    _need(v_cache, "v_cache", None, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seqlens, "seqlens", torch.int32, 1)
    _need(k_scale, "k_scale", torch.float32)
    _need(v_scale, "v_scale", torch.float32)
    if k_cache.dtype != v_cache.dtype or k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache must match")
    bs, h_q, hd = q.shape
    num_blocks, h_kv, page, hd2 = k_cache.shape
    if hd2 != hd:
        raise ValueError("head_dim mismatch")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(hd)
    if max_seqlen is None:
        max_seqlen = block_table.shape[1] * page
    splits = gqa_num_splits(bs, h_kv, max_seqlen, num_splits)
    if out is None:
        out = torch.empty((bs, h_q, hd), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((bs, h_q), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = gqa_workspace_bytes(bs, h_q, hd, splits)
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=q.device)
    _check(lib().paged_gqa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), kv_dtype_code(k_cache), num_blocks,
                                  _ptr(k_scale), _ptr(v_scale), _ptr(block_table), block_table.shape[1],
                                  _ptr(seqlens), float(softmax_scale), splits, _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse),
                                  bs, h_q, h_kv, hd, page, _stream(q.device)),
           "paged_gqa_decode")
    return out, lse


def paged_gqa_decode_ext(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                         block_table: torch.Tensor, seqlens: torch.Tensor, k_scale: torch.Tensor,
                         v_scale: torch.Tensor, softmax_scale: float | None = None, spec_mask=None,
                         window: int = 0, sinks=None, num_splits: int = 0, max_seqlen: int | None = None,
                         out=None, lse=None, workspace=None):
    """Paged GQA decode with per-row scales and the XQA options.  q bf16 [bs, q_len, h_q, hd]
    (the sequence's last q_len cache positions); k_scale / v_scale float32 [1] or per cached row
    [num_blocks, h_kv, page]; spec_mask uint8 [bs, q_len, q_len] or None (causal inside the
    block); window 0 = off; sinks float32 [h_q] or None.  Returns (out bf16 [bs, q_len, h_q, hd],
    lse [bs, q_len, h_q])."""
    _need(q, "q", torch.bfloat16, 4)
    _need(k_cache, "k_cache", None, 4)
    _need(v_cache, "v_cache", None, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seqlens, "seqlens", torch.int32, 1)
    _need(k_scale, "k_scale", torch.float32)
    _need(v_scale, "v_scale", torch.float32)
    if k_cache.dtype != v_cache.dtype or k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache must match")
    bs, q_len, h_q, hd = q.shape
    num_blocks, h_kv, page, hd2 = k_cache.shape
    if hd2 != hd:
        raise ValueError("head_dim mismatch")
    per_row = k_scale.numel() != 1 or v_scale.numel() != 1
    if per_row and (tuple(k_scale.shape) != (num_blocks, h_kv, page) or tuple(v_scale.shape) != (num_blocks, h_kv, page)):
        raise ValueError("per-row scales must both be [num_blocks, h_kv, page]")
    if spec_mask is not None:
        _need(spec_mask, "spec_mask", torch.uint8, 3)
        if tuple(spec_mask.shape) != (bs, q_len, q_len):
            raise ValueError("spec_mask must be [bs, q_len, q_len]")
    if sinks is not None:
        _need(sinks, "sinks", torch.float32, 1)
        if sinks.numel() != h_q:
            raise ValueError("sinks must be [h_q]")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(hd)
    if max_seqlen is None:
        max_seqlen = block_table.shape[1] * page
    splits = gqa_ext_num_splits(bs, h_kv, max_seqlen, q_len, window, num_splits)
    if out is None:
        out = torch.empty((bs, q_len, h_q, hd), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((bs, q_len, h_q), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = gqa_workspace_bytes(bs, h_q, hd, splits)
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=q.device)
    _check(lib().paged_gqa_decode_ext(_ptr(q), _ptr(k_cache), _ptr(v_cache), kv_dtype_code(k_cache), num_blocks,
                                      _ptr(k_scale), _ptr(v_scale), 1 if per_row else 0, _ptr(block_table),
                                      block_table.shape[1], _ptr(seqlens), float(softmax_scale), q_len,
                                      _ptr(spec_mask), int(window), _ptr(sinks), splits, _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse),
                                      bs, h_q, h_kv, hd, page, _stream(q.device)),
           "paged_gqa_decode_ext")
    return out, lse


# ------------------------------------------------------------ cache write --


def paged_cache_write(x: torch.Tensor, slot_mapping: torch.Tensor, cache: torch.Tensor, *,
                      tensor_scale: torch.Tensor | None = None,
                      token_scales: torch.Tensor | None = None) -> None:
    """Quantise bf16 rows into an E4M3 paged cache, in place.

    cache E4M3 (or uint8) [num_blocks, h_kv, page, head_dim] with x bf16
    [n_tokens, h_kv, head_dim], or the dense MLA form [num_pages, page, d]
    with x [n_tokens, d].  slot_mapping int32 [n_tokens] (block * page +
    offset; negative = skip).  Exactly one of tensor_scale (float32 [1]) or
    token_scales (float32 [num_blocks, h_kv, page], written per row) is given.
    x may be strided along tokens; each token's rows must be contiguous."""
    if cache.dim() == 3:
        cache4 = cache.unsqueeze(1)
        x3 = x.unsqueeze(1) if x.dim() == 2 else x
    else:
        cache4, x3 = cache, x
    if not x3.is_cuda or x3.dtype != torch.bfloat16 or x3.dim() != 3:
        raise ValueError("x must be a CUDA bf16 tensor [n_tokens, h_kv, head_dim] (or [n_tokens, d])")
    _need(cache4, "cache", None, 4)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    num_blocks, h_kv, page, hd = cache4.shape
    n_tokens = x3.shape[0]
    if tuple(x3.shape[1:]) != (h_kv, hd) or slot_mapping.shape[0] != n_tokens:
        raise ValueError("x, slot_mapping and cache shapes disagree")
    if x3.stride(2) != 1 or (h_kv > 1 and x3.stride(1) != hd):
        raise ValueError("each token's rows of x must be contiguous")
    if tensor_scale is not None:
        _need(tensor_scale, "tensor_scale", torch.float32)
    if token_scales is not None:
        _need(token_scales, "token_scales", torch.float32)
        if tuple(token_scales.shape) != (num_blocks, h_kv, page):
            raise ValueError("token_scales must be [num_blocks, h_kv, page]")
    _check(lib().fp8_paged_cache_write(_ptr(x3), x3.stride(0) if n_tokens > 0 else h_kv * hd,
                                       _ptr(slot_mapping), n_tokens, h_kv, hd, page, num_blocks,
                                       kv_dtype_code(cache4), _ptr(cache4), _ptr(tensor_scale),
                                       _ptr(token_scales), _stream(x3.device)),
           "fp8_paged_cache_write")


def wait_timeout_site(device=None):
    """(source line, block, thread) of the first dense-MLA bounded wait that ran out
    since the last call, or None (synchronises the current stream; clears the record)."""
    where = (ctypes.c_uint32 * 3)()
    _check(lib().fp8mla_get_wait_timeout_site(_stream(device), where), "fp8mla_get_wait_timeout_site")
    return None if where[0] == 0 else (where[0], where[1], where[2])


def set_wait_test(fault_page: int = 0, wait_limit_ns: int = 0) -> None:
    """Test hook of the bounded waits of the FP8-dots MLA decode (current device):
    fault_page = p + 1 makes CTA 0 of work unit 0 skip the loads of its p-th page,
    so its waits run out (0 = off); wait_limit_ns replaces the wait limit (0 = default)."""
    _check(lib().fp8mla_set_wait_test(int(fault_page), int(wait_limit_ns)), "fp8mla_set_wait_test")


def set_stage_timing(enable: bool) -> None:
    """Measurement aid: while enabled, ``decode`` records events between its kernels
    (which stops them overlapping); ``stage_times`` then reads the last call's stages."""
    _check(lib().fp8mla_set_stage_timing(1 if enable else 0), "fp8mla_set_stage_timing")


def stage_times(device=None):
    """(Q quantisation, decode kernel, combine) milliseconds of the last timed ``decode``
    call (synchronises the current stream)."""
    ms = (ctypes.c_float * 3)()
    _check(lib().fp8mla_get_stage_times(_stream(device), ms), "fp8mla_get_stage_times")
    return ms[0], ms[1], ms[2]


def last_device_error(device=None) -> int:
    """OR of the device status bits since the last call (synchronises the current stream)."""
    code = ctypes.c_uint32(0)
    _check(lib().fp8mla_get_last_device_error(_stream(device), ctypes.byref(code)),
           "fp8mla_get_last_device_error")
    return code.value
