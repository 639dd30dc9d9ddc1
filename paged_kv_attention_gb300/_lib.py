"""ctypes view of libpagedattn.so: the C ABI declared in include/paged_attn.h, nothing more."""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpagedattn.so")

PA_OK = 0
PA_ERR_INVALID_ARGUMENT = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_WORKSPACE_TOO_SMALL = 3
PA_ERR_CUDA = 4

PA_DTYPE_F32 = 0
PA_DTYPE_BF16 = 1
PA_DTYPE_INT8 = 2
PA_DTYPE_FP8_E4M3 = 3

PA_SHORT_AUTO = 0
PA_SHORT_SPLIT = 1
PA_SHORT_TENSOR = 2

PA_ERRBIT_PAGE_OUT_OF_POOL = 1
PA_ERRBIT_LENGTH_OUT_OF_RANGE = 2
PA_ERRBIT_SLOT_OUT_OF_POOL = 4
PA_ERRBIT_QUERY_LAYOUT = 8
PA_ERRBIT_WAIT_TIMEOUT = 16

_i, _f, _p, _sz = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t


class AttnOptions(ctypes.Structure):
    """pa_attn_options: sliding window, logit softcap, device pointer to per-head sink logits."""
    _fields_ = [("sliding_window", ctypes.c_int32), ("logit_softcap", ctypes.c_float), ("sinks", ctypes.c_void_p)]


_opt = ctypes.POINTER(AttnOptions)


class RowStrides(ctypes.Structure):
    """pa_row_strides: elements from one q row / out row to the next (0 = dense)."""
    _fields_ = [("q", ctypes.c_int64), ("out", ctypes.c_int64)]


_rs = ctypes.POINTER(RowStrides)
_i64 = ctypes.c_int64

# name -> (restype, argtypes); mirrors include/paged_attn.h
SIGNATURES = {
    "pa_status_string": (ctypes.c_char_p, [_i]),
    "pa_version": (_i, []),
    "pa_supports": (_i, [_i, _i, _i, _i, _i, _i]),
    "pa_plan_decode_splits": (_i, [_i, _i, _i, _i, _i]),
    "pa_decode_auto_splits": (_i, [_i, _i, _i, _i, _i, _i, _i]),
    "pa_decode_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "pa_reshape_and_cache": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p]),
    "pa_paged_attention_decode": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _i, _i,
                                       _p, _p, _sz, _p, _p]),
    "pa_paged_attention_varlen": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                       _i, _f, _i, _p, _p, _p]),
    "pa_paged_attention_decode_static_scratch": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f,
                                                      _i, _i, _p, _p, _p]),
    "pa_paged_attention_decode_ex": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _i, _i,
                                          _p, _p, _sz, _opt, _p, _p]),
    "pa_selftest_wait_timeout": (_i, [_i, _p, _p]),
    "pa_cascade_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "pa_cascade_decode": (_i, [_p, _p, _p, _p, _p, _i, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _i, _p, _p, _sz,
                               _p, _p]),
    "pa_reshape_and_cache_quant": (_i, [_p, _p, _i, _p, _p, _p, _p, _i, _p, _i, _i, _i, _i, _i, _p, _p]),
    "pa_paged_attention_decode_quant": (_i, [_p, _p, _p, _p, _p, _i, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f,
                                             _i, _p, _p, _sz, _opt, _p, _p]),
    "pa_paged_attention_varlen_quant": (_i, [_p, _p, _p, _p, _p, _i, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i,
                                             _i, _i, _i, _f, _p, _opt, _p, _p]),
    "pa_paged_attention_varlen_ex": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                          _i, _f, _i, _p, _opt, _p, _p]),
    "pa_paged_attention_varlen_ws": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                          _i, _f, _i, _p, _opt, _p, _sz, _p, _p]),
    "pa_varlen_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "pa_reshape_and_cache_strided": (_i, [_p, _p, _i64, _i64, _p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p]),
    "pa_paged_attention_decode_strided": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _i, _i,
                                               _p, _p, _sz, _opt, _rs, _p, _p]),
    "pa_paged_attention_varlen_strided": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                               _i, _f, _i, _p, _opt, _rs, _p, _sz, _p, _p]),
    "pa_varlen_plan_capacity": (_i, [_i, _i, _i, _i]),
    "pa_varlen_plan": (_i, [_p, _p, _i, _i, _i, _i, _i, _i, _i, _p, _i]),
    "pa_paged_attention_varlen_planned": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                               _i, _f, _i, _p, _opt, _rs, _p, _sz, _p, _i, _p, _p]),
    "pa_paged_attention_varlen_sched": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                             _i, _f, _i, _p, _opt, _rs, _i, _p, _sz, _p, _p]),
}

_lib = None


class LibraryMissing(RuntimeError):
    pass


def load() -> ctypes.CDLL:
    """Load the in-tree library (built by ``paged_kv_attention_gb300.build``). Raises if absent:
    there is no fallback implementation."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise LibraryMissing(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
