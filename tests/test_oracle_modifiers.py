"""Pins for the oracle's sliding window, logit softcap and attention sinks: hand-derived closed
forms (tests/golden/score_modifiers_tiny.json), invariants, and a library special case (a sink
is an extra key of zero value: torch SDPA with an additive mask)."""

import json
import math
import os

import torch
import torch.nn.functional as F

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "score_modifiers_tiny.json")


def _g():
    with open(GOLDEN) as f:
        return json.load(f)


def _pool(keys, values, bs=2):
    L = len(keys)
    n = workloads.cdiv(L, bs)
    kc = torch.full((n, bs, 1, 1), float("nan"), dtype=torch.float64)
    vc = kc.clone()
    for p in range(L):
        kc[p // bs, p % bs, 0, 0] = keys[p]
        vc[p // bs, p % bs, 0, 0] = values[p]
    return kc, vc, torch.arange(n, dtype=torch.int32)[None, :]


def test_golden_softcap():
    c = _g()["softcap"]
    cap = c["cap"]
    keys = [cap * math.atanh(math.log(3.0) / cap) if k == "cap_atanh_ln3" else k for k in c["keys"]]
    kc, vc, t = _pool(keys, c["values"])
    q = torch.ones((1, 1, 1), dtype=torch.float64)
    out = oracle.paged_attention_decode(q, kc, vc, t, torch.tensor([2], dtype=torch.int32), 1.0, softcap=cap)
    assert abs(float(out[0, 0, 0]) - c["expected"]) < 1e-12


def test_golden_sink():
    c = _g()["sink"]
    keys = [math.log(2.0) if k == "ln2" else k for k in c["keys"]]
    kc, vc, t = _pool(keys, c["values"])
    q = torch.ones((1, 1, 1), dtype=torch.float64)
    sinks = torch.tensor([math.log(3.0)], dtype=torch.float64)
    out = oracle.paged_attention_decode(q, kc, vc, t, torch.tensor([2], dtype=torch.int32), 1.0, sinks=sinks)
    assert abs(float(out[0, 0, 0]) - c["expected"]) < 1e-12


def test_golden_window():
    c = _g()["window"]
    kc, vc, t = _pool(c["keys"], c["values"])
    q = torch.zeros((1, 1, 1), dtype=torch.float64)
    for w, want in c["expected"].items():
        out = oracle.paged_attention_decode(q, kc, vc, t, torch.tensor([3], dtype=torch.int32), 1.0, window=int(w))
        assert abs(float(out[0, 0, 0]) - want) < 1e-12


def _case(seed, q_lens, seq_lens, hq=4, hkv=2, d=8, bs=4):
    need = sum(workloads.cdiv(L, bs) for L in seq_lens)
    case = workloads.make_case("m", seed, q_lens, seq_lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                               block_size=bs, dtype=torch.float64, pool_blocks=need + 2, table_multiple=4)
    kc, vc = case.empty_pools()
    oracle.reshape_and_cache(case.key, case.value, kc, vc, case.slot_mapping)
    return case, kc, vc


def _varlen(case, kc, vc, **kw):
    return oracle.paged_attention_varlen(case.q, kc, vc, case.query_start_loc, case.seq_lens, case.block_tables,
                                         True, case.scale, **kw)


def test_window_covering_everything_changes_nothing():
    case, kc, vc = _case(1, [5, 1, 9], [12, 30, 9])
    assert torch.equal(_varlen(case, kc, vc), _varlen(case, kc, vc, window=30))


def test_window_one_returns_own_value():
    case, kc, vc = _case(2, [6, 1], [6, 17])
    out = _varlen(case, kc, vc, window=1)
    off, qsl = 0, case.query_start_loc.tolist()
    for r, L in enumerate(case.seq_lens.tolist()):
        q_len = qsl[r + 1] - qsl[r]
        for t in range(q_len):
            v = case.value[off + L - q_len + t].double()                        # the query's own position
            assert torch.allclose(out[qsl[r] + t], v.repeat_interleave(2, dim=0), rtol=0, atol=1e-14)
        off += L


def test_decode_window_equals_decode_of_the_last_positions():
    w = 7
    case, kc, vc = _case(3, [1, 1], [20, 9])
    got = oracle.paged_attention_decode(case.q, kc, vc, case.block_tables, case.seq_lens, case.scale, window=w)
    # the last w positions of each sequence, laid into a fresh pool from position 0
    off = 0
    for s, L in enumerate(case.seq_lens.tolist()):
        keep = min(w, L)
        sub = workloads.make_case("sub", 9, [1], [keep], num_q_heads=4, num_kv_heads=2, head_dim=8, block_size=4,
                                  dtype=torch.float64, table_multiple=4)
        sub.key = case.key[off + L - keep: off + L]
        sub.value = case.value[off + L - keep: off + L]
        skc, svc = sub.empty_pools()
        oracle.reshape_and_cache(sub.key, sub.value, skc, svc, sub.slot_mapping)
        want = oracle.paged_attention_decode(case.q[s:s + 1], skc, svc, sub.block_tables, sub.seq_lens, case.scale)
        assert torch.allclose(got[s], want[0], rtol=0, atol=1e-14)
        off += L


def test_huge_softcap_changes_nothing_and_sink_at_minus_infinity_changes_nothing():
    case, kc, vc = _case(4, [3, 1], [10, 25])
    base = _varlen(case, kc, vc)
    assert torch.allclose(_varlen(case, kc, vc, softcap=1e9), base, rtol=0, atol=1e-12)
    sinks = torch.full((4,), -math.inf, dtype=torch.float64)
    assert torch.allclose(_varlen(case, kc, vc, sinks=sinks), base, rtol=0, atol=1e-15)


def test_softcap_bounds_the_scores():
    # scaled scores far beyond the cap behave like exactly +-cap: with all scores equal to
    # +huge they tie, so the result is the mean of the values
    case, kc, vc = _case(5, [1], [11], hq=2, hkv=2, d=8)
    q = torch.full_like(case.q, 50.0)
    kc.copy_(torch.where(torch.isnan(kc), kc, torch.full_like(kc, 50.0)))
    out = oracle.paged_attention_varlen(q, kc, vc, case.query_start_loc, case.seq_lens, case.block_tables, True,
                                        case.scale, softcap=3.0)
    mean = case.value.double().mean(0)
    assert torch.allclose(out[0], mean, rtol=0, atol=1e-12)


def test_sinks_equal_a_zero_value_key_in_torch_sdpa():
    L, D, hq, hkv = 13, 8, 4, 2
    case, kc, vc = _case(6, [L], [L], hq=hq, hkv=hkv, d=D)
    sinks = torch.tensor([0.3, -1.2, 2.0, 0.0], dtype=torch.float64)
    got = _varlen(case, kc, vc, sinks=sinks)
    G = hq // hkv
    q = case.q.double().permute(1, 0, 2)[None]                                   # [1, Hq, L, D]
    k = case.key.double().repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    v = case.value.double().repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    # one extra key per head with q.k = 0 and value 0, whose logit the additive mask sets to the sink
    k = torch.cat([k, torch.zeros_like(k[:, :, :1])], dim=2)
    v = torch.cat([v, torch.zeros_like(v[:, :, :1])], dim=2)
    mask = torch.full((1, hq, L, L + 1), -math.inf, dtype=torch.float64)
    causal = torch.tril(torch.ones(L, L, dtype=torch.bool))
    mask[..., :L] = torch.where(causal, 0.0, -math.inf)
    mask[..., L] = sinks[None, :, None]
    want = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=case.scale)[0].permute(1, 0, 2)
    assert torch.allclose(got, want, rtol=0, atol=1e-12)


def test_window_matches_torch_sdpa_band_mask():
    L, w = 21, 5
    case, kc, vc = _case(7, [L], [L], hq=4, hkv=4, d=8)
    got = _varlen(case, kc, vc, window=w)
    q = case.q.double().permute(1, 0, 2)[None]
    k = case.key.double().permute(1, 0, 2)[None]
    v = case.value.double().permute(1, 0, 2)[None]
    band = torch.tril(torch.ones(L, L, dtype=torch.bool)) & torch.triu(torch.ones(L, L, dtype=torch.bool), -(w - 1))
    want = F.scaled_dot_product_attention(q, k, v, attn_mask=band, scale=case.scale)[0].permute(1, 0, 2)
    assert torch.allclose(got, want, rtol=0, atol=1e-12)
