"""Pins for the 8-bit KV cache oracle (oracle/quant.py): the hand-derived golden quantisation,
the error bound the definition implies, the code range edge, the write/gather round trip, the
accuracy of attention over the dequantised cache against full precision, a hand-derived golden
of attention over int8 / E4M3 codes, and exact agreement of both 8-bit attention functions with
the plain oracle over a float64 pool of code * scale (with planted slips shown to fail)."""

import json
import math
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


# --------------------------------------------------------------------------- exact pins
# "32. Production attention kernels", Quantized KV caches: the kernel multiplies the tile of
# codes by its per-slot scale and then attends to it exactly like a bf16 tile. Attention over an
# 8-bit cache is therefore the plain definition applied to a float64 pool holding code * scale;
# both products are exact in float64, so the two oracles must agree to the last bit (<= 1e-15).

def _golden_quant_pools(g, kind):
    """The golden's code and scale pools ([3, 2, 1, 1] codes, [3, 2, 1] scales)."""
    def codes(rows):
        return [[[[1.0 if c == "unused" else float(c)]] for c in row] for row in rows]

    def scales(rows):
        return [[[float("nan") if s == "nan" else float(s)] for s in row] for row in rows]
    kc = torch.tensor(codes(g["k_codes"]), dtype=torch.float32).to(quant.CODE_DTYPE[kind])
    vc = torch.tensor(codes(g["v_codes"]), dtype=torch.float32).to(quant.CODE_DTYPE[kind])
    ks = torch.tensor(scales(g["k_scales"]), dtype=torch.float32)
    vs = torch.tensor(scales(g["v_scales"]), dtype=torch.float32)
    return kc, vc, ks, vs


@pytest.mark.parametrize("kind", ["int8", "fp8"])
def test_golden_quantized_attention(kind):
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "attention_quant_tiny.json")))
    kc, vc, ks, vs = _golden_quant_pools(g, kind)
    # every golden code is exact in the code format
    assert kc.float()[:, :, 0, 0].tolist()[1] == [0.0, 4.0] and vc.float()[0, 0, 0, 0].item() == 44.0
    scale = math.log(3.0)
    q = torch.tensor(g["q"], dtype=torch.float64)[:, None, None]          # [3, 1, 1]
    qsl = torch.tensor(g["query_start_loc"], dtype=torch.int32)
    lens = torch.tensor(g["seq_lens"], dtype=torch.int32)
    tables = torch.tensor(g["block_tables"], dtype=torch.int32)
    for causal, key in ((True, "expected_causal"), (False, "expected_noncausal")):
        out = quant.paged_attention_varlen_quant(q, kc, vc, ks, vs, qsl, lens, tables, causal=causal, scale=scale)
        assert torch.isfinite(out).all()
        assert [round(float(x), 12) for x in out[:, 0, 0]] == g[key], (causal, out[:, 0, 0].tolist())
    dec = quant.paged_attention_decode_quant(q[1:2], kc, vc, ks, vs, tables[:1], lens[:1], scale=scale)
    assert abs(float(dec[0, 0, 0]) - g["expected_decode_seq0"]) < 1e-12


def _dequantised_pool(codes, scales):
    """float64 pool of code * scale, computed here elementwise over the whole pool."""
    return codes.to(torch.float64) * scales.to(torch.float64)[..., None]


def _quant_case(kind, q_lens, seq_lens, seed, hq=8, hkv=2, d=16, bs=4):
    need = sum(workloads.cdiv(L, bs) for L in seq_lens)
    case = workloads.make_case("qpin", seed, q_lens, seq_lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                               block_size=bs, dtype=torch.bfloat16, pool_blocks=need + 3, table_multiple=4)
    shape = (case.num_blocks, bs, hkv, d)
    kc = torch.zeros(shape, dtype=quant.CODE_DTYPE[kind])
    vc = torch.zeros(shape, dtype=quant.CODE_DTYPE[kind])
    ks = torch.zeros(shape[:3], dtype=torch.float32)
    vs = torch.zeros(shape[:3], dtype=torch.float32)
    quant.reshape_and_cache_quant(case.key, case.value, kc, vc, ks, vs, case.slot_mapping, kind)
    # the scales of the keys and the values of one slot differ (their rows differ), so a swap shows
    return case, kc, vc, ks, vs


MODIFIERS = [dict(), dict(window=7), dict(softcap=0.9), dict(sinks=torch.tensor([0.5, -2.0, 3.0, 0.0] * 2)),
             dict(window=3, softcap=2.0, sinks=torch.tensor([1.0] * 8))]


@pytest.mark.parametrize("kind", ["int8", "fp8"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("mod", range(len(MODIFIERS)))
def test_varlen_quant_equals_plain_oracle_on_dequantised_pool(kind, causal, mod):
    # q_len 0, 1, 5 and 37 against contexts that cross several pages (bs 4) and end mid-page
    case, kc, vc, ks, vs = _quant_case(kind, [0, 1, 5, 37], [9, 23, 14, 41], seed=40 + mod)
    kw = MODIFIERS[mod]
    got = quant.paged_attention_varlen_quant(case.q, kc, vc, ks, vs, case.query_start_loc, case.seq_lens,
                                             case.block_tables, causal=causal, scale=case.scale, **kw)
    want = oracle.paged_attention_varlen(case.q, _dequantised_pool(kc, ks), _dequantised_pool(vc, vs),
                                         case.query_start_loc, case.seq_lens, case.block_tables, causal,
                                         case.scale, **kw)
    assert (got - want).abs().max().item() <= 1e-15


@pytest.mark.parametrize("kind", ["int8", "fp8"])
@pytest.mark.parametrize("mod", range(len(MODIFIERS)))
def test_decode_quant_equals_plain_oracle_on_dequantised_pool(kind, mod):
    case, kc, vc, ks, vs = _quant_case(kind, [1, 1, 1, 1], [1, 17, 30, 0], seed=60 + mod)
    kw = MODIFIERS[mod]
    got = quant.paged_attention_decode_quant(case.q, kc, vc, ks, vs, case.block_tables, case.seq_lens,
                                             case.scale, **kw)
    want = oracle.paged_attention_decode(case.q, _dequantised_pool(kc, ks), _dequantised_pool(vc, vs),
                                         case.block_tables, case.seq_lens, case.scale, **kw)
    assert (got - want).abs().max().item() <= 1e-15
    assert torch.equal(got[3], torch.zeros_like(got[3]))  # empty context


def test_quant_pins_catch_planted_mistakes(monkeypatch):
    """The two exact pins above fail on the slips they are meant to catch, planted in the oracle."""
    kind = "int8"
    case, kc, vc, ks, vs = _quant_case(kind, [0, 1, 5, 37], [9, 23, 14, 41], seed=40)
    plain = oracle.paged_attention_varlen(case.q, _dequantised_pool(kc, ks), _dequantised_pool(vc, vs),
                                          case.query_start_loc, case.seq_lens, case.block_tables, True, case.scale)

    def run():
        return quant.paged_attention_varlen_quant(case.q, kc, vc, ks, vs, case.query_start_loc, case.seq_lens,
                                                  case.block_tables, causal=True, scale=case.scale)
    assert (run() - plain).abs().max().item() <= 1e-15
    # 1. key and value scales swapped
    swapped = quant.paged_attention_varlen_quant(case.q, kc, vc, vs, ks, case.query_start_loc, case.seq_lens,
                                                 case.block_tables, causal=True, scale=case.scale)
    assert (swapped - plain).abs().max().item() > 1e-3
    # 2. a position rule of q_pos = t (the request's first query at position 0)
    real_attend = quant.attend
    monkeypatch.setattr(quant, "attend", lambda q_rows, q_pos, *a, **k: real_attend(q_rows, q_pos - q_pos.min(),
                                                                                    *a, **k))
    assert (run() - plain).abs().max().item() > 1e-3
    monkeypatch.setattr(quant, "attend", real_attend)
    # 3. the scale of the next slot (an off-by-one in the scale gather)
    real_deq = quant.dequantized_context
    monkeypatch.setattr(quant, "dequantized_context",
                        lambda c, s, t, n: real_deq(c, torch.roll(s, 1, dims=1), t, n))
    assert (run() - plain).abs().max().item() > 1e-3
