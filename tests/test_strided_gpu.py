"""GPU checks of the row-strided entry points (pa_*_strided): the queries and the new keys and
values as slices of a fused QKV projection output, the output as a slice of a wider buffer.

A strided call runs the dense call's arithmetic on other addresses, so its result must equal the
dense call's bit for bit (the dense calls' parity with the float64 oracle is what the other GPU
files check); one case per path is also held to the oracle, and the heads of the wider output
buffer outside the slice must keep their sentinel values."""

import pytest
import torch

import oracle
import paged_kv_attention_gb300 as pa
import workloads
from paged_helpers import check_close, gpu_pools, oracle_pools

pytestmark = pytest.mark.gpu
DEV = "cuda"
SENTINEL = -7.0


def fused_qkv(case):
    """[N, Hq + 2 Hkv, D] buffer holding q in its first Hq heads; returns (buffer, q view)."""
    n, hq, d = case.q.shape
    buf = torch.full((n, hq + 2 * case.num_kv_heads, d), 3.0, dtype=case.q.dtype, device=DEV)
    buf[:, :hq] = case.q.to(DEV)
    return buf, buf[:, :hq]


def wide_out(like, pad_heads=8):
    """[N, Hq + pad, D] sentinel buffer and its [N, Hq, D] slice starting pad/2 heads in."""
    n, hq, d = like.shape
    buf = torch.full((n, hq + pad_heads, d), SENTINEL, dtype=like.dtype, device=DEV)
    off = pad_heads // 2
    return buf, buf[:, off:off + hq]


def untouched(buf, view_heads, pad_heads=8):
    off = pad_heads // 2
    outside = torch.cat([buf[:, :off], buf[:, off + view_heads:]], dim=1)
    return bool((outside == SENTINEL).all())


def decode_case(seed, lens, hq, hkv, d, bs, dtype):
    return workloads.decode_case("strided", seed, lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                 block_size=bs, dtype=dtype)


@pytest.mark.parametrize("d,hq,hkv,dtype", [(128, 32, 8, torch.bfloat16), (64, 8, 2, torch.bfloat16),
                                            (256, 16, 4, torch.bfloat16), (64, 8, 2, torch.float32),
                                            (128, 16, 16, torch.float32)])
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_decode_strided_equals_dense(d, hq, hkv, dtype, splits):
    case = decode_case(900 + d + hq + splits, [1, 17, 200, 1000, 64], hq, hkv, d, 16, dtype)
    kc, vc = gpu_pools(case)
    t, lens = case.block_tables.to(DEV), case.seq_lens.to(DEV)
    dense = pa.paged_attention_decode(case.q.to(DEV), kc, vc, t, lens, case.scale, num_splits=splits)
    _, qv = fused_qkv(case)
    obuf, ov = wide_out(qv)
    got = pa.paged_attention_decode(qv, kc, vc, t, lens, case.scale, num_splits=splits, out=ov)
    assert got.data_ptr() == ov.data_ptr()
    assert torch.equal(ov, dense)
    assert untouched(obuf, hq)


def test_decode_strided_against_oracle():
    case = decode_case(931, [5, 300, 2049], 32, 8, 128, 16, torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    _, qv = fused_qkv(case)
    obuf, ov = wide_out(qv)
    pa.paged_attention_decode(qv, kc, vc, case.block_tables.to(DEV), case.seq_lens.to(DEV), case.scale, out=ov)
    want = oracle.paged_attention_decode(case.q, ko, vo, case.block_tables, case.seq_lens, case.scale)
    check_close(ov, want, torch.bfloat16, label="strided decode")


def varlen_case(seed, q_lens, seq_lens, hq, hkv, d, bs, dtype):
    return workloads.make_case("strided_varlen", seed, q_lens, seq_lens, num_q_heads=hq, num_kv_heads=hkv,
                               head_dim=d, block_size=bs, dtype=dtype)


VARLEN_SHAPES = [(128, 32, 8, 16, torch.bfloat16),   # tensor-core kernel
                 (128, 16, 2, 64, torch.bfloat16),   # tensor-core kernel, group 8
                 (64, 8, 2, 16, torch.bfloat16),     # tensor-core kernel at head_dim 64
                 (256, 16, 4, 32, torch.bfloat16),   # the head_dim-256 tensor-core kernel
                 (128, 8, 8, 16, torch.float32)]     # fp32: one-split decode per token


@pytest.mark.parametrize("d,hq,hkv,bs,dtype", VARLEN_SHAPES)
@pytest.mark.parametrize("split_decodes", [False, True, "tensor"])
def test_varlen_strided_equals_dense(d, hq, hkv, bs, dtype, split_decodes):
    """(split_decodes "tensor": the device-planned grid with every request on the tensor cores.)"""
    if split_decodes == "tensor":
        if dtype != torch.bfloat16:
            pytest.skip("schedules are a bf16 tensor-core feature")
        kw = dict(schedule="tensor")
    else:
        kw = dict(split_decodes=split_decodes)
    q_lens = [1, 5, 37, 130, 1, 0, 64]
    seq_lens = [700, 5, 37, 900, 1, 3, 200]
    case = varlen_case(950 + d + hq + bs, q_lens, seq_lens, hq, hkv, d, bs, dtype)
    kc, vc = gpu_pools(case)
    args = (kc, vc, case.query_start_loc.to(DEV), case.seq_lens.to(DEV), case.block_tables.to(DEV), max(q_lens))
    dense = pa.paged_attention_varlen(case.q.to(DEV), *args, True, case.scale, **kw)
    _, qv = fused_qkv(case)
    obuf, ov = wide_out(qv)
    pa.paged_attention_varlen(qv, *args, True, case.scale, out=ov, **kw)
    assert torch.equal(ov, dense)
    assert untouched(obuf, hq)


def test_varlen_strided_against_oracle():
    q_lens, seq_lens = [1, 5, 300], [1500, 900, 300]
    case = varlen_case(977, q_lens, seq_lens, 32, 8, 128, 16, torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    _, qv = fused_qkv(case)
    obuf, ov = wide_out(qv)
    pa.paged_attention_varlen(qv, kc, vc, case.query_start_loc.to(DEV), case.seq_lens.to(DEV),
                              case.block_tables.to(DEV), max(q_lens), True, case.scale, out=ov)
    want = oracle.paged_attention_varlen(case.q, ko, vo, case.query_start_loc, case.seq_lens, case.block_tables,
                                         causal=True, scale=case.scale)
    check_close(ov, want, torch.bfloat16, label="strided varlen")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_cache_write_from_fused_rows_is_bit_exact(dtype):
    case = varlen_case(990, [1, 1], [300, 77], 8, 2, 128, 16, dtype)
    t, hkv, d = case.key.shape
    # rows of a fused [T, Hq + 2 Hkv, D] projection output: K after the 8 query heads, then V
    fused = torch.randn(t, 8 + 2 * hkv, d, device=DEV).to(dtype)
    fused[:, 8:8 + hkv] = case.key.to(DEV)
    fused[:, 8 + hkv:] = case.value.to(DEV)
    kv, vv = fused[:, 8:8 + hkv], fused[:, 8 + hkv:]
    assert not kv.is_contiguous()
    kc, vc = (x.to(DEV) for x in case.empty_pools())
    pa.reshape_and_cache(kv, vv, kc, vc, case.slot_mapping.to(DEV))
    kd, vd = gpu_pools(case)
    assert torch.equal(kc.view(torch.int32 if dtype == torch.float32 else torch.int16),
                       kd.view(torch.int32 if dtype == torch.float32 else torch.int16))
    assert torch.equal(vc.view(torch.int32 if dtype == torch.float32 else torch.int16),
                       vd.view(torch.int32 if dtype == torch.float32 else torch.int16))


def test_bad_row_strides_are_refused():
    case = decode_case(995, [10, 20], 8, 2, 128, 16, torch.bfloat16)
    kc, vc = gpu_pools(case)
    t, lens = case.block_tables.to(DEV), case.seq_lens.to(DEV)
    # rows 8 * 128 + 4 elements apart: 8-byte steps break the 16-byte row alignment
    store = torch.zeros(2 * (8 * 128 + 4), dtype=torch.bfloat16, device=DEV)
    qv = store.as_strided((2, 8, 128), (8 * 128 + 4, 128, 1))
    with pytest.raises(pa.PagedAttentionError):
        pa.paged_attention_decode(qv, kc, vc, t, lens, case.scale)
    # heads not dense within a row: refused by the binding before the C call
    with pytest.raises(ValueError):
        pa.paged_attention_decode(case.q.to(DEV).transpose(0, 1).contiguous().transpose(0, 1), kc, vc, t, lens,
                                  case.scale)
