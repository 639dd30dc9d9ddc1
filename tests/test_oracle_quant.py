"""Pins for the 8-bit KV cache oracle (oracle/quant.py): the hand-derived golden quantisation,
the error bound the definition implies, the code range edge, the write/gather round trip, and
the accuracy of attention over the dequantised cache against full precision."""

import json
import os

import pytest
import torch

import oracle
from oracle import quant
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quantize_kv_tiny.json")


def test_golden_quantization():
    g = json.load(open(GOLDEN))
    x = torch.tensor(g["x"], dtype=torch.float32)
    codes, scales = quant.quantize_kv(x, "int8")
    assert codes.tolist() == g["int8_codes"]
    assert torch.equal(scales, torch.tensor(g["amax"], dtype=torch.float32) / 127.0)
    codes, scales = quant.quantize_kv(x, "fp8")
    assert codes.float().tolist() == g["fp8_codes"]
    assert torch.equal(scales, torch.tensor(g["amax"], dtype=torch.float32) / 448.0)


@pytest.mark.parametrize("kind", ["int8", "fp8"])
def test_range_edge_and_error_bound(kind):
    x = torch.randn((300, 4, 64), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    codes, scales = quant.quantize_kv(x, kind)
    c = codes.to(torch.float64)
    qmax = quant.Q_MAX[kind]
    # the largest |x| of each (token, head) lands on the code range's edge
    assert torch.allclose(c.abs().amax(-1), torch.full_like(c[..., 0], qmax))
    deq = c * scales.double()[..., None]
    err = (deq - x.double()).abs()
    if kind == "int8":
        assert (err <= scales.double()[..., None] * (0.5 + 1e-5)).all()   # half a step
    else:
        # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 (plus the subnormal floor)
        assert (err <= x.double().abs() * 2.0 ** -4 + scales.double()[..., None] * 2.0 ** -10).all()


@pytest.mark.parametrize("kind", ["int8", "fp8"])
def test_write_then_gather_round_trip(kind):
    case = workloads.make_case("q", 5, [1, 1], [37, 20], num_q_heads=4, num_kv_heads=2, head_dim=16, block_size=4,
                               dtype=torch.bfloat16, pool_blocks=20, table_multiple=4)
    shape = (case.num_blocks, case.block_size, 2, 16)
    kc = torch.zeros(shape, dtype=quant.CODE_DTYPE[kind])
    vc = torch.zeros(shape, dtype=quant.CODE_DTYPE[kind])
    ks = torch.zeros(shape[:3], dtype=torch.float32)
    vs = torch.zeros(shape[:3], dtype=torch.float32)
    quant.reshape_and_cache_quant(case.key, case.value, kc, vc, ks, vs, case.slot_mapping, kind)
    codes, scales = quant.quantize_kv(case.key, kind)
    want = codes.to(torch.float64) * scales.double()[..., None]
    off = 0
    for r, L in enumerate(case.seq_lens.tolist()):
        got = quant.dequantized_context(kc, ks, case.block_tables[r], L)
        assert torch.equal(got, want[off:off + L])
        off += L


@pytest.mark.parametrize("kind,tol", [("int8", 2e-2), ("fp8", 8e-2)])
def test_quantized_attention_stays_close_to_full_precision(kind, tol):
    case = workloads.decode_case("qa", 6, [50, 400, 1], num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
                                 dtype=torch.bfloat16)
    kc, vc = case.empty_pools()
    oracle.reshape_and_cache(case.key, case.value, kc, vc, case.slot_mapping)
    full = oracle.paged_attention_decode(case.q, kc, vc, case.block_tables, case.seq_lens, case.scale)
    shape = kc.shape
    qk = torch.zeros(shape, dtype=quant.CODE_DTYPE[kind])
    qv = torch.zeros(shape, dtype=quant.CODE_DTYPE[kind])
    ks = torch.zeros(shape[:3], dtype=torch.float32)
    vs = torch.zeros(shape[:3], dtype=torch.float32)
    quant.reshape_and_cache_quant(case.key, case.value, qk, qv, ks, vs, case.slot_mapping, kind)
    got = quant.paged_attention_decode_quant(case.q, qk, qv, ks, vs, case.block_tables, case.seq_lens, case.scale)
    assert (got - full).abs().max().item() < tol
    # a single cached position returns its dequantised value exactly
    assert torch.allclose(got[2], quant.dequantized_context(qv, vs, case.block_tables[2], 1)[0].repeat_interleave(4, 0),
                          rtol=0, atol=1e-15)
