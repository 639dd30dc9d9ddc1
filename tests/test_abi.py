"""Host-side checks of the C ABI: the library loads without a GPU, exports every symbol the
header declares, and its host logic (status strings, split planning, workspace sizing,
argument refusal before any launch) behaves as documented. No kernel is launched."""

import ctypes
import os
import re

import pytest

from paged_kv_attention_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    from paged_kv_attention_gb300 import build
    if build.is_stale():
        build.build()
    return _lib.load()


def declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("pa_reshape_and_cache", "pa_paged_attention_decode", "pa_paged_attention_varlen",
                     "pa_decode_workspace_bytes", "pa_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and the binding's table covers them all
    assert set(declared_functions()) <= set(_lib.SIGNATURES)


def test_status_strings(lib):
    assert lib.pa_status_string(0) == b"PA_OK"
    assert lib.pa_status_string(3) == b"PA_ERR_WORKSPACE_TOO_SMALL"
    assert lib.pa_status_string(99) == b"PA_ERR_UNKNOWN"
    assert lib.pa_version() >= 100


def test_supports(lib):
    bf16, f32 = _lib.PA_DTYPE_BF16, _lib.PA_DTYPE_F32
    assert lib.pa_supports(0, 128, 32, 8, 16, bf16)
    assert lib.pa_supports(1, 256, 16, 4, 64, bf16)
    assert lib.pa_supports(0, 64, 8, 2, 16, f32)
    assert not lib.pa_supports(0, 96, 8, 2, 16, bf16)      # head_dim
    assert not lib.pa_supports(0, 128, 32, 8, 8, bf16)     # bf16 needs block_size % 16 == 0
    assert lib.pa_supports(0, 128, 32, 8, 8, f32)
    assert not lib.pa_supports(0, 128, 12, 8, 16, bf16)    # Hq % Hkv
    assert not lib.pa_supports(0, 256, 16, 1, 16, f32)     # group * D > 2048
    assert not lib.pa_supports(0, 128, 64, 2, 16, bf16)    # group 32


class TestSplitPlanning:
    """pa_plan_decode_splits: the choose_splits rule of "32. Production attention kernels"
    (Long contexts: split the keys) with a preferred shortest split and a whole-wave criterion."""

    def test_degenerate_inputs_give_one(self, lib):
        assert lib.pa_plan_decode_splits(0, 10, 152, 3, 64) == 1
        assert lib.pa_plan_decode_splits(4, 0, 152, 3, 64) == 1
        assert lib.pa_plan_decode_splits(4, 10, 0, 3, 64) == 1

    def test_bounds(self, lib):
        for units in (1, 2, 8, 32, 256, 512, 4096):
            for chunks in (1, 3, 4, 13, 64, 256, 2048):
                for min_chunks in (0, 4, 64, 256):
                    s = lib.pa_plan_decode_splits(units, chunks, 152, 3, min_chunks)
                    assert 1 <= s <= 32
                    assert s <= max(1, chunks // 4)          # no split under 4 chunks

    def test_small_batch_long_context_splits(self, lib):
        # 1 sequence x 2 KV heads over 256 chunks: long splits cannot fill 152 SMs, so split
        # down to one full wave (capped at 32)
        assert lib.pa_plan_decode_splits(2, 256, 152, 3, 64) >= 16
        assert lib.pa_plan_decode_splits(32, 256, 152, 2, 256) == 10   # 320 CTAs >= 304 slots

    def test_long_splits_fill_waves(self, lib):
        # 64 x 8 units over 256 chunks at 3 CTAs/SM: splits of >= 64 chunks allow 1-4; 4 fills
        # its 5 waves best (90%)
        s = lib.pa_plan_decode_splits(512, 256, 152, 3, 64)
        assert s == 4
        assert 256 // s >= 64

    def test_enough_ctas_stay_whole(self, lib):
        # one wave of CTAs already, and splits must cover >= 256 chunks: no split
        assert lib.pa_plan_decode_splits(512, 256, 152, 2, 256) == 1

    def test_short_contexts_do_not_split(self, lib):
        assert lib.pa_plan_decode_splits(4096, 4, 152, 3, 64) == 1


def test_workspace_bytes(lib):
    f = lib.pa_decode_workspace_bytes
    assert f(4, 32, 128, 16, 16, 1) == 0                                 # one split: none
    assert f(4, 32, 128, 16, 16, 3) == 4 * 3 * 32 * 130 * 4
    assert f(4, 32, 128, 256, 16, 0) == 4 * 32 * 32 * 130 * 4            # auto: bound over any choice
    assert f(4, 32, 128, 2, 16, 8) == 4 * 2 * 32 * 130 * 4               # never more splits than chunks
    assert f(0, 32, 128, 16, 16, 0) == 0


def test_varlen_workspace_bytes(lib):
    f = lib.pa_varlen_workspace_bytes

    def plan(reqs, max_q):  # the device-planned work list: reqs * cdiv(max_q, 16) int32, 256-byte rounded
        return -(-(reqs * -(-max_q // 16) * 4) // 256) * 256
    # then the short requests' partials: 8 query rows each, at most 8 splits (never more than the
    # 16-token chunks)
    assert f(64, 32, 128, 256, 16) == plan(64, 4096) + 64 * 8 * 8 * 32 * 130 * 4
    assert f(4, 8, 64, 2, 16) == plan(4, 32) + 4 * 8 * 2 * 8 * 66 * 4     # 2 chunks: at most 2 splits
    assert f(4, 8, 64, 1, 16) == plan(4, 16)                            # one chunk: one split, no partials
    assert f(0, 8, 64, 16, 16) == 0


def _decode_args(**over):
    a = dict(q=16, k=16, v=16, tables=16, lens=16, S=1, Hq=8, Hkv=2, D=128, bs=16, nb=4, mb=16,
             scale=0.0, dtype=_lib.PA_DTYPE_BF16, splits=0, out=16, ws=None, ws_bytes=0, err=None, stream=None)
    a.update(over)
    return [a[k] for k in ("q", "k", "v", "tables", "lens", "S", "Hq", "Hkv", "D", "bs", "nb", "mb", "scale",
                           "dtype", "splits", "out", "ws", "ws_bytes", "err", "stream")]


@pytest.mark.parametrize("over,status", [
    (dict(q=None), _lib.PA_ERR_INVALID_ARGUMENT),
    (dict(lens=None), _lib.PA_ERR_INVALID_ARGUMENT),
    (dict(Hq=6, Hkv=4), _lib.PA_ERR_INVALID_ARGUMENT),
    (dict(S=-1), _lib.PA_ERR_INVALID_ARGUMENT),
    (dict(splits=33), _lib.PA_ERR_INVALID_ARGUMENT),
    (dict(scale=-1.0), _lib.PA_ERR_INVALID_ARGUMENT),
    (dict(scale=float("nan")), _lib.PA_ERR_INVALID_ARGUMENT),
    (dict(q=8), _lib.PA_ERR_INVALID_ARGUMENT),               # misaligned pointer
    (dict(D=96), _lib.PA_ERR_UNSUPPORTED),
    (dict(bs=8), _lib.PA_ERR_UNSUPPORTED),                   # bf16 needs 16-token chunks
    (dict(Hq=64, Hkv=2), _lib.PA_ERR_UNSUPPORTED),           # group 32
    (dict(dtype=7), _lib.PA_ERR_UNSUPPORTED),
    (dict(S=0), _lib.PA_OK),                                 # nothing to do, nothing launched
])
def test_decode_refuses_bad_arguments_before_launch(lib, over, status):
    assert lib.pa_paged_attention_decode(*_decode_args(**over)) == status


def test_varlen_and_cache_write_refuse_bad_arguments(lib):
    bf16 = _lib.PA_DTYPE_BF16
    # pa_paged_attention_varlen(q,k,v,qsl,seq_lens,tables, R,N,maxq, Hq,Hkv,D,bs,nb,mb, causal,scale,dtype,out,err,stream)
    ok_args = [16, 16, 16, 16, 16, 16, 2, 5, 4, 8, 2, 128, 16, 4, 16, 1, 0.0, bf16, 16, None, None]
    bad_qsl = list(ok_args)
    bad_qsl[3] = None
    assert lib.pa_paged_attention_varlen(*bad_qsl) == _lib.PA_ERR_INVALID_ARGUMENT
    bad_d = list(ok_args)
    bad_d[11] = 80
    assert lib.pa_paged_attention_varlen(*bad_d) == _lib.PA_ERR_UNSUPPORTED
    empty = list(ok_args)
    empty[7] = 0
    assert lib.pa_paged_attention_varlen(*empty) == _lib.PA_OK
    # pa_reshape_and_cache(key,value,kc,vc,slots, N,Hkv,D,bs,nb,dtype,err,stream)
    assert lib.pa_reshape_and_cache(16, 16, 16, 16, None, 3, 2, 128, 16, 4, bf16, None, None) == \
        _lib.PA_ERR_INVALID_ARGUMENT
    assert lib.pa_reshape_and_cache(16, 16, 16, 16, 16, 3, 2, 128, 16, 4, 9, None, None) == _lib.PA_ERR_UNSUPPORTED
    assert lib.pa_reshape_and_cache(16, 16, 16, 16, 16, 0, 2, 128, 16, 4, bf16, None, None) == _lib.PA_OK
    assert lib.pa_reshape_and_cache(16, 16, 16, 16, 16, 3, 1, 4, 16, 4, bf16, None, None) == \
        _lib.PA_ERR_UNSUPPORTED                                       # 8-byte rows


# a layout that passes the stride checks stops at the next one: the workspace (with a GPU) or the
# device query (without one); neither launches anything
PASSED = (_lib.PA_ERR_WORKSPACE_TOO_SMALL, _lib.PA_ERR_CUDA)


@pytest.mark.parametrize("q_stride,out_stride,status", [
    (0, 0, PASSED),
    (8 * 128 + 64, 0, PASSED),
    (8 * 128 - 8, 0, _lib.PA_ERR_INVALID_ARGUMENT),   # rows would overlap
    (0, 8 * 128 + 4, _lib.PA_ERR_INVALID_ARGUMENT),   # 8-byte rows: not a whole 16-byte unit
    (-8, 0, _lib.PA_ERR_INVALID_ARGUMENT),
])
def test_strided_calls_check_row_strides_before_launch(lib, q_stride, out_stride, status):
    # two sequences and 4 splits: the dense layout reaches the workspace check (no launch)
    args = _decode_args(S=2, splits=4)
    st = _lib.RowStrides(q_stride, out_stride)
    got = lib.pa_paged_attention_decode_strided(*args[:18], None, ctypes.byref(st), None, None)
    assert got in status if isinstance(status, tuple) else got == status
    bf16 = _lib.PA_DTYPE_BF16
    # pa_paged_attention_varlen_strided(q,k,v,qsl,lens,tables, R,N,maxq, Hq,Hkv,D,bs,nb,mb, causal,scale,dtype,
    #                                   out,options,strides,ws,ws_bytes,err,stream)
    if status == _lib.PA_ERR_INVALID_ARGUMENT:
        v = [16, 16, 16, 16, 16, 16, 2, 5, 4, 8, 2, 128, 16, 4, 16, 1, 0.0, bf16, 16, None, ctypes.byref(st),
             None, 0, None, None]
        assert lib.pa_paged_attention_varlen_strided(*v) == status
    # key/value row strides of the cache write: Hkv * D = 256 elements dense
    assert lib.pa_reshape_and_cache_strided(16, 16, 255, 0, 16, 16, 16, 3, 2, 128, 16, 4, bf16, None, None) == \
        _lib.PA_ERR_INVALID_ARGUMENT
    assert lib.pa_reshape_and_cache_strided(16, 16, 0, 260, 16, 16, 16, 3, 2, 128, 16, 4, bf16, None, None) == \
        _lib.PA_ERR_INVALID_ARGUMENT
    assert lib.pa_reshape_and_cache_strided(16, 16, 264, 0, 16, 16, 16, 0, 2, 128, 16, 4, bf16, None, None) == \
        _lib.PA_OK                                                    # no tokens: nothing launched


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(_lib.LibraryMissing):
        _lib.load()
    assert isinstance(ctypes.CDLL, type)
