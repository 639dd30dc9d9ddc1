"""Paged KV attention for GB300 (sm_103a): a thin Python binding over libpagedattn.so.

The functions below only marshal torch tensors into the C ABI of
``include/paged_attn.h`` (pointers, sizes, the current CUDA stream) and turn a
non-OK status into an exception. Every step of the computation runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback, and calling any of
them without the built library raises.
"""

from __future__ import annotations

import ctypes
import math

import torch

from . import _lib

__all__ = [
    "PagedAttentionError",
    "cascade_decode",
    "decode_auto_splits",
    "decode_workspace_bytes",
    "plan_decode_splits",
    "paged_attention_decode",
    "paged_attention_varlen",
    "paged_attention_decode_quant",
    "paged_attention_varlen_quant",
    "reshape_and_cache_quant",
    "reshape_and_cache",
    "status_string",
    "supports",
]

_DTYPES = {torch.bfloat16: _lib.PA_DTYPE_BF16, torch.float32: _lib.PA_DTYPE_F32}


class PagedAttentionError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {status_string(status)}")
        self.status = status


def status_string(status: int) -> str:
    return _lib.load().pa_status_string(int(status)).decode()


def _dtype(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise PagedAttentionError("dtype", _lib.PA_ERR_UNSUPPORTED) from None


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the C ABI must be contiguous")
    return t.data_ptr()


def _row_ptr(t: torch.Tensor) -> tuple[int, int]:
    """(data pointer, row stride in elements) of a [rows, heads, D] tensor whose heads and head
    dims are dense and whose rows may sit further apart (e.g. a slice of a fused QKV output)."""
    if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
        raise ValueError("rows of [rows, heads, head_dim] must hold their heads densely")
    if t.shape[0] > 1 and t.stride(0) < t.shape[1] * t.shape[2]:
        raise ValueError("rows must not overlap")
    return t.data_ptr(), (t.stride(0) if t.shape[0] > 1 else t.shape[1] * t.shape[2])


def _strides(q: torch.Tensor, out: torch.Tensor):
    """pa_row_strides for the *_strided calls, or None when q and out are dense."""
    if q.is_contiguous() and out.is_contiguous():
        return None
    return ctypes.byref(_lib.RowStrides(_row_ptr(q)[1], _row_ptr(out)[1]))


def _stream(stream: torch.cuda.Stream | None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(fn: str, status: int) -> None:
    if status != _lib.PA_OK:
        raise PagedAttentionError(fn, status)


def supports(is_varlen: bool, head_dim: int, num_q_heads: int, num_kv_heads: int, block_size: int,
             dtype: torch.dtype) -> bool:
    return bool(_lib.load().pa_supports(int(is_varlen), head_dim, num_q_heads, num_kv_heads, block_size,
                                        _DTYPES.get(dtype, -1)))


def plan_decode_splits(num_units: int, max_chunks: int, num_sms: int, ctas_per_sm: int,
                       min_chunks_per_split: int = 64) -> int:
    return _lib.load().pa_plan_decode_splits(num_units, max_chunks, num_sms, ctas_per_sm, min_chunks_per_split)


def decode_auto_splits(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                       max_blocks_per_seq: int, dtype: torch.dtype) -> int:
    """Split count an auto decode call with these sizes uses on the current device (0 = refused)."""
    return _lib.load().pa_decode_auto_splits(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                             max_blocks_per_seq, _DTYPES.get(dtype, -1))


def decode_workspace_bytes(num_seqs: int, num_q_heads: int, head_dim: int, max_blocks_per_seq: int,
                           block_size: int, num_splits: int = 0) -> int:
    return int(_lib.load().pa_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_blocks_per_seq,
                                                     block_size, num_splits))


def _options(window: int, softcap: float, sinks: torch.Tensor | None):
    """pa_attn_options for the *_ex calls, or None when no modifier is asked for."""
    if not window and not softcap and sinks is None:
        return None
    if sinks is not None and (sinks.dtype != torch.float32 or not sinks.is_cuda):
        raise ValueError("sinks must be a float32 CUDA tensor of num_q_heads logits")
    return ctypes.byref(_lib.AttnOptions(int(window), float(softcap), _ptr(sinks)))


def reshape_and_cache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      slot_mapping: torch.Tensor, error_word: torch.Tensor | None = None,
                      stream: torch.cuda.Stream | None = None) -> None:
    """k_cache[slot // bs, slot % bs] = key[i] for slot = slot_mapping[i] >= 0 (same for v).
    key and value may be row-strided views (heads dense within a row)."""
    n, hkv, d = key.shape
    nb, bs = k_cache.shape[0], k_cache.shape[1]
    if key.is_contiguous() and value.is_contiguous():
        st = _lib.load().pa_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                              _ptr(slot_mapping), n, hkv, d, bs, nb, _dtype(key),
                                              _ptr(error_word), _stream(stream))
        _check("pa_reshape_and_cache", st)
        return
    (kp, ks), (vp, vs) = _row_ptr(key), _row_ptr(value)
    st = _lib.load().pa_reshape_and_cache_strided(kp, vp, ks, vs, _ptr(k_cache), _ptr(v_cache),
                                                  _ptr(slot_mapping), n, hkv, d, bs, nb, _dtype(key),
                                                  _ptr(error_word), _stream(stream))
    _check("pa_reshape_and_cache_strided", st)


def paged_attention_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor,
                           scale: float | None = None, num_splits: int = 0,
                           out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                           error_word: torch.Tensor | None = None,
                           stream: torch.cuda.Stream | None = None, window: int = 0, softcap: float = 0.0,
                           sinks: torch.Tensor | None = None) -> torch.Tensor:
    """One query per sequence over its paged context (split-KV + combine in the library).

    ``workspace`` (a byte or fp32 CUDA tensor) is allocated here when not given; pass one
    to keep the call allocation-free (e.g. under CUDA-graph capture). ``window``,
    ``softcap`` and ``sinks`` are the pa_attn_options score modifiers."""
    s, hq, d = q.shape
    nb, bs, hkv = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    mb = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    ws_bytes = decode_workspace_bytes(s, hq, d, mb, bs, num_splits)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    strides = _strides(q, out)
    if strides is None:
        st = _lib.load().pa_paged_attention_decode_ex(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
            s, hq, hkv, d, bs, nb, mb, float(scale or 0.0), _dtype(q), int(num_splits),
            _ptr(out), _ptr(workspace), ws_len, _options(window, softcap, sinks), _ptr(error_word),
            _stream(stream))
    else:
        st = _lib.load().pa_paged_attention_decode_strided(
            _row_ptr(q)[0], _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
            s, hq, hkv, d, bs, nb, mb, float(scale or 0.0), _dtype(q), int(num_splits),
            _row_ptr(out)[0], _ptr(workspace), ws_len, _options(window, softcap, sinks), strides,
            _ptr(error_word), _stream(stream))
    _check("pa_paged_attention_decode", st)
    return out


SHORT_REQUEST_QUERIES = 8  # requests of at most this many queries go to the split-KV decode


def varlen_plan(query_start_loc: torch.Tensor, seq_lens: torch.Tensor, max_query_len: int, num_q_heads: int,
                num_kv_heads: int, causal: bool = True, window: int = 0, split_decodes: bool = False) -> torch.Tensor:
    """Host plan of the tensor-core grid for one batch (pa_varlen_plan): the (tile pair, request)
    items that exist, longest first, as a CPU int32 tensor to copy to the device and pass as
    ``work_items``. ``split_decodes`` must match the call's."""
    qsl = query_start_loc.to("cpu", torch.int32).contiguous()
    sl = seq_lens.to("cpu", torch.int32).contiguous()
    r = sl.shape[0]
    lib = _lib.load()
    cap = int(lib.pa_varlen_plan_capacity(r, int(max_query_len), num_q_heads, num_kv_heads))
    if cap < 0:
        raise PagedAttentionError("pa_varlen_plan_capacity", _lib.PA_ERR_INVALID_ARGUMENT)
    items = torch.empty(max(cap, 1), dtype=torch.int32)
    n = int(lib.pa_varlen_plan(qsl.data_ptr(), sl.data_ptr(), r, int(max_query_len), num_q_heads, num_kv_heads,
                               int(bool(causal)), int(window), SHORT_REQUEST_QUERIES if split_decodes else 0,
                               items.data_ptr(), cap))
    if n < 0:
        raise PagedAttentionError("pa_varlen_plan", _lib.PA_ERR_INVALID_ARGUMENT)
    return items[:n]


def paged_attention_varlen(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           query_start_loc: torch.Tensor, seq_lens: torch.Tensor,
                           block_tables: torch.Tensor, max_query_len: int, causal: bool = True,
                           scale: float | None = None, out: torch.Tensor | None = None,
                           error_word: torch.Tensor | None = None,
                           stream: torch.cuda.Stream | None = None, window: int = 0, softcap: float = 0.0,
                           sinks: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                           split_decodes: bool = False, work_items: torch.Tensor | None = None,
                           schedule: str | None = None) -> torch.Tensor:
    """Flattened prefill / verify / decode batch; request r's queries are the newest q_len of
    its seq_lens[r] positions, causal by position. ``window``, ``softcap`` and ``sinks`` are
    the pa_attn_options score modifiers.

    ``schedule`` (pa_paged_attention_varlen_sched; a workspace is allocated unless one is given):
    "auto", "split" or "tensor" run the tensor-core kernel on a grid planned on the device (only
    the tile pairs the batch has, longest first; graph-safe), with the short requests (1 to 8
    queries) on the split-KV decode for "split", on the tensor-core kernel for "tensor", and for
    "auto" on the split-KV decode when the batch has >= 80 requests averaging <= 8 queries.
    Without ``schedule``: ``work_items`` (a host plan, see varlen_plan) or the default grid, with
    ``split_decodes`` sending the short requests to the split-KV decode."""
    n, hq, d = q.shape
    nb, bs, hkv = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    r = seq_lens.shape[0]
    mb = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    lib = _lib.load()
    modes = {"auto": _lib.PA_SHORT_AUTO, "split": _lib.PA_SHORT_SPLIT, "tensor": _lib.PA_SHORT_TENSOR}
    if split_decodes and schedule is None and work_items is None:
        schedule = "split"
    if schedule is not None and schedule not in modes:
        raise ValueError(f"schedule must be one of {sorted(modes)}")
    if (split_decodes or schedule is not None) and q.dtype == torch.bfloat16 and workspace is None:
        workspace = torch.empty(max(int(lib.pa_varlen_workspace_bytes(r, hq, d, mb, bs)), 16), dtype=torch.uint8,
                                device=q.device)
    if schedule is None and not split_decodes:
        workspace = None
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    strides = _strides(q, out)
    if schedule is not None:
        if work_items is not None:
            raise ValueError("schedule plans on the device: pass no work_items")
        st = lib.pa_paged_attention_varlen_sched(
            _row_ptr(q)[0], _ptr(k_cache), _ptr(v_cache), _ptr(query_start_loc), _ptr(seq_lens),
            _ptr(block_tables), r, n, int(max_query_len), hq, hkv, d, bs, nb, mb, int(bool(causal)),
            float(scale or 0.0), _dtype(q), _row_ptr(out)[0], _options(window, softcap, sinks), strides,
            modes[schedule], _ptr(workspace), ws_len, _ptr(error_word), _stream(stream))
    elif work_items is not None:
        if work_items.dtype != torch.int32 or not work_items.is_cuda:
            raise ValueError("work_items must be an int32 CUDA tensor (varlen_plan's output, copied)")
        st = lib.pa_paged_attention_varlen_planned(
            _row_ptr(q)[0], _ptr(k_cache), _ptr(v_cache), _ptr(query_start_loc), _ptr(seq_lens),
            _ptr(block_tables), r, n, int(max_query_len), hq, hkv, d, bs, nb, mb, int(bool(causal)),
            float(scale or 0.0), _dtype(q), _row_ptr(out)[0], _options(window, softcap, sinks), strides,
            _ptr(workspace), ws_len, _ptr(work_items) if work_items.numel() else 16, int(work_items.numel()),
            _ptr(error_word), _stream(stream))
    elif strides is None:
        st = lib.pa_paged_attention_varlen_ws(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(query_start_loc), _ptr(seq_lens), _ptr(block_tables),
            r, n, int(max_query_len), hq, hkv, d, bs, nb, mb, int(bool(causal)), float(scale or 0.0),
            _dtype(q), _ptr(out), _options(window, softcap, sinks), _ptr(workspace), ws_len, _ptr(error_word),
            _stream(stream))
    else:
        st = lib.pa_paged_attention_varlen_strided(
            _row_ptr(q)[0], _ptr(k_cache), _ptr(v_cache), _ptr(query_start_loc), _ptr(seq_lens),
            _ptr(block_tables), r, n, int(max_query_len), hq, hkv, d, bs, nb, mb, int(bool(causal)),
            float(scale or 0.0), _dtype(q), _row_ptr(out)[0], _options(window, softcap, sinks), strides,
            _ptr(workspace), ws_len, _ptr(error_word), _stream(stream))
    _check("pa_paged_attention_varlen", st)
    return out


def cascade_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, prefix_table: torch.Tensor,
                   prefix_len: torch.Tensor, suffix_tables: torch.Tensor, suffix_lens: torch.Tensor,
                   scale: float | None = None, num_splits: int = 0, out: torch.Tensor | None = None,
                   workspace: torch.Tensor | None = None, error_word: torch.Tensor | None = None,
                   stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Decode of S sequences that share a cached prefix (``prefix_len``: a device int32 scalar)
    followed by their own suffixes; the prefix K/V is read once for all of them."""
    s, hq, d = q.shape
    nb, bs, hkv = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    mb = suffix_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    lib = _lib.load()
    if workspace is None:
        workspace = torch.empty(max(int(lib.pa_cascade_workspace_bytes(s, hq, d, bs, prefix_table.numel(), mb)), 16),
                                dtype=torch.uint8, device=q.device)
    ws_len = workspace.numel() * workspace.element_size()
    st = lib.pa_cascade_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(prefix_table), _ptr(prefix_len),
                               prefix_table.numel(), _ptr(suffix_tables), _ptr(suffix_lens), s, hq, hkv, d, bs, nb,
                               mb, float(scale or 0.0), int(num_splits), _ptr(out), _ptr(workspace), ws_len,
                               _ptr(error_word), _stream(stream))
    _check("pa_cascade_decode", st)
    return out


# ----------------------------------------------------------------------------- 8-bit caches
_CODES = {torch.int8: _lib.PA_DTYPE_INT8, torch.float8_e4m3fn: _lib.PA_DTYPE_FP8_E4M3}


def _cache_kind(t: torch.Tensor) -> int:
    try:
        return _CODES[t.dtype]
    except KeyError:
        raise PagedAttentionError("cache dtype", _lib.PA_ERR_UNSUPPORTED) from None


def reshape_and_cache_quant(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            k_scales: torch.Tensor, v_scales: torch.Tensor, slot_mapping: torch.Tensor,
                            error_word: torch.Tensor | None = None,
                            stream: torch.cuda.Stream | None = None) -> None:
    """Quantise key/value rows (bf16 or fp32) into int8 / fp8 code pools plus per-(slot, head)
    fp32 scales, through the slot mapping."""
    n, hkv, d = key.shape
    nb, bs = k_cache.shape[0], k_cache.shape[1]
    st = _lib.load().pa_reshape_and_cache_quant(
        _ptr(key), _ptr(value), _dtype(key), _ptr(k_cache), _ptr(v_cache), _ptr(k_scales), _ptr(v_scales),
        _cache_kind(k_cache), _ptr(slot_mapping), n, hkv, d, bs, nb, _ptr(error_word), _stream(stream))
    _check("pa_reshape_and_cache_quant", st)


def paged_attention_decode_quant(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                 k_scales: torch.Tensor, v_scales: torch.Tensor, block_tables: torch.Tensor,
                                 context_lens: torch.Tensor, scale: float | None = None, num_splits: int = 0,
                                 out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                                 error_word: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None,
                                 window: int = 0, softcap: float = 0.0,
                                 sinks: torch.Tensor | None = None) -> torch.Tensor:
    """Decode over an int8 / fp8 cache (q, out bf16)."""
    s, hq, d = q.shape
    nb, bs, hkv = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    mb = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    ws_bytes = decode_workspace_bytes(s, hq, d, mb, bs, num_splits)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _lib.load().pa_paged_attention_decode_quant(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scales), _ptr(v_scales), _cache_kind(k_cache),
        _ptr(block_tables), _ptr(context_lens), s, hq, hkv, d, bs, nb, mb, float(scale or 0.0), int(num_splits),
        _ptr(out), _ptr(workspace), ws_len, _options(window, softcap, sinks), _ptr(error_word), _stream(stream))
    _check("pa_paged_attention_decode_quant", st)
    return out


def paged_attention_varlen_quant(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                 k_scales: torch.Tensor, v_scales: torch.Tensor, query_start_loc: torch.Tensor,
                                 seq_lens: torch.Tensor, block_tables: torch.Tensor, max_query_len: int,
                                 causal: bool = True, scale: float | None = None, out: torch.Tensor | None = None,
                                 error_word: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None,
                                 window: int = 0, softcap: float = 0.0,
                                 sinks: torch.Tensor | None = None) -> torch.Tensor:
    """Varlen attention over an int8 / fp8 cache (q, out bf16)."""
    n, hq, d = q.shape
    nb, bs, hkv = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    r = seq_lens.shape[0]
    mb = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    st = _lib.load().pa_paged_attention_varlen_quant(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scales), _ptr(v_scales), _cache_kind(k_cache),
        _ptr(query_start_loc), _ptr(seq_lens), _ptr(block_tables), r, n, int(max_query_len), hq, hkv, d, bs, nb, mb,
        int(bool(causal)), float(scale or 0.0), _ptr(out), _options(window, softcap, sinks), _ptr(error_word),
        _stream(stream))
    _check("pa_paged_attention_varlen_quant", st)
    return out


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
