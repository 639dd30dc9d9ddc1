"""Pins for the float64 oracle: it is checked against things other than itself.

Each pin is chosen so that a plausible slip in the oracle (a swapped page/row
index, the wrong KV head for a query head, a wrong causal offset, a dropped
normalisation or scale) fails at least one of them:

* closed forms: one visible position returns its value; equal scores return
  the mean; a constant V returns that constant; an empty context returns zeros
  ("paged-attn-xpu", Validation); the hand-derived golden softmax cases;
* a brute-force pool scan in pure Python that enumerates pool slots (not
  positions) and finds each slot's position through the block table;
* a special case that is a library routine: torch SDPA (float64, is_causal for
  full prefill) on a contiguous cache, GQA expanded by repeat_interleave;
* invariants: page permutation, GQA == repeat_kv, chunked prefill == full
  prefill row by row, varlen with q_len 1 == decode;
* reshape_and_cache: the hand-written golden fixture and a write/gather round trip.
"""

import json
import math
import os

import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _filled_pools(case):
    kc, vc = case.empty_pools()
    oracle.reshape_and_cache(case.key, case.value, kc, vc, case.slot_mapping)
    return kc, vc


def _tiny_varlen(seed, q_lens, seq_lens, hq=4, hkv=2, d=8, bs=4, dtype=torch.float64, pool_extra=3):
    need = sum(workloads.cdiv(L, bs) for L in seq_lens)
    return workloads.make_case("tiny", seed, q_lens, seq_lens, num_q_heads=hq, num_kv_heads=hkv,
                               head_dim=d, block_size=bs, dtype=dtype, pool_blocks=need + pool_extra,
                               table_multiple=4)


# --------------------------------------------------------------------------- closed forms

def test_single_position_returns_its_value():
    case = _tiny_varlen(1, [1, 1], [1, 1])
    kc, vc = _filled_pools(case)
    out = oracle.paged_attention_decode(case.q, kc, vc, case.block_tables, case.seq_lens, case.scale)
    G = case.num_q_heads // case.num_kv_heads
    for s in range(2):
        for h in range(case.num_q_heads):
            page = int(case.block_tables[s, 0])
            assert torch.equal(out[s, h], vc[page, 0, h // G].double())


def test_equal_scores_give_the_mean():
    case = _tiny_varlen(2, [1, 1, 1], [7, 13, 4])
    case.q.zero_()
    kc, vc = _filled_pools(case)
    out = oracle.paged_attention_decode(case.q, kc, vc, case.block_tables, case.seq_lens, case.scale)
    G = case.num_q_heads // case.num_kv_heads
    off = 0
    for s, L in enumerate(case.seq_lens.tolist()):
        vals = case.value[off:off + L].double()          # tokens in position order
        off += L
        for h in range(case.num_q_heads):
            assert torch.allclose(out[s, h], vals[:, h // G].mean(0), rtol=0, atol=1e-13)


def test_constant_values_return_the_constant():
    case = _tiny_varlen(3, [3, 1], [9, 22])
    case.value.fill_(0.375)
    kc, vc = _filled_pools(case)
    out = oracle.paged_attention_varlen(case.q, kc, vc, case.query_start_loc, case.seq_lens,
                                        case.block_tables, True, case.scale)
    assert torch.allclose(out, torch.full_like(out, 0.375), rtol=0, atol=1e-14)


def test_empty_context_gives_zeros():
    case = _tiny_varlen(4, [1, 1], [0, 5])
    kc, vc = _filled_pools(case)
    out = oracle.paged_attention_decode(case.q, kc, vc, case.block_tables, case.seq_lens, case.scale)
    assert torch.equal(out[0], torch.zeros_like(out[0]))
    assert torch.isfinite(out).all()


def _golden_pool(keys, values, block_size):
    """[L] scalar keys/values -> single-head, head_dim-1 pool laid out in page order."""
    L = len(keys)
    n_pages = workloads.cdiv(L, block_size)
    kc = torch.full((n_pages, block_size, 1, 1), float("nan"), dtype=torch.float64)
    vc = kc.clone()
    for p in range(L):
        kc[p // block_size, p % block_size, 0, 0] = keys[p]
        vc[p // block_size, p % block_size, 0, 0] = values[p]
    table = torch.arange(n_pages, dtype=torch.int32)[None, :]
    return kc, vc, table


def test_golden_softmax_weights():
    g = _load("softmax_weights_tiny.json")["cases"]
    c = g["weights"]
    keys = [math.log(3.0) if k == "ln3" else k for k in c["keys"]]
    kc, vc, table = _golden_pool(keys, c["values"], c["block_size"])
    q = torch.tensor([[c["q"]]], dtype=torch.float64)                     # [1, 1, 1]
    out = oracle.paged_attention_decode(q, kc, vc, table, torch.tensor([2], dtype=torch.int32), c["scale"])
    assert abs(float(out[0, 0, 0]) - c["expected"]) < 1e-13


def test_golden_causal_position_rule():
    c = _load("softmax_weights_tiny.json")["cases"]["causal_offset"]
    kc, vc, table = _golden_pool(c["keys"], c["values"], c["block_size"])
    q = torch.tensor(c["q"], dtype=torch.float64)[:, None, :]             # [2, 1, 1]
    qsl = torch.tensor([0, 2], dtype=torch.int32)
    out = oracle.paged_attention_varlen(q, kc, vc, qsl, torch.tensor([3], dtype=torch.int32), table,
                                        True, c["scale"])
    assert [round(float(x), 12) for x in out[:, 0, 0]] == c["expected"]


# --------------------------------------------------------------------------- brute force

def _brute_force_pool_scan(case, kc, vc, causal):
    """Pure-Python, slot-driven: visit every pool slot, find which request
    position (if any) it holds by looking the page up in the request's table."""
    N, Hq, D = case.q.shape
    Hkv = case.num_kv_heads
    G = Hq // Hkv
    bs = case.block_size
    out = [[[0.0] * D for _ in range(Hq)] for _ in range(N)]
    qsl = case.query_start_loc.tolist()
    for r, L in enumerate(case.seq_lens.tolist()):
        q_len = qsl[r + 1] - qsl[r]
        n_pages = -(-L // bs)
        table = case.block_tables[r, :n_pages].tolist()
        for t in range(q_len):
            my_pos = L - q_len + t
            for h in range(Hq):
                entries = []
                for b in range(kc.shape[0]):
                    if b not in table:
                        continue
                    page_index = table.index(b)
                    for o in range(bs):
                        p = page_index * bs + o
                        if p >= L or (causal and p > my_pos):
                            continue
                        kv = h // G
                        qk = sum(float(case.q[qsl[r] + t, h, d]) * float(kc[b, o, kv, d]) for d in range(D))
                        entries.append((case.scale * qk, [float(vc[b, o, kv, d]) for d in range(D)]))
                if not entries:
                    continue
                mx = max(e[0] for e in entries)
                wsum = sum(math.exp(e[0] - mx) for e in entries)
                for d in range(D):
                    out[qsl[r] + t][h][d] = sum(math.exp(e[0] - mx) * e[1][d] for e in entries) / wsum
    return torch.tensor(out, dtype=torch.float64)


@pytest.mark.parametrize("hq,hkv,bs", [(4, 2, 4), (3, 1, 2), (4, 4, 1), (6, 2, 4)])
@pytest.mark.parametrize("causal", [True, False])
def test_brute_force_pool_scan(hq, hkv, bs, causal):
    case = _tiny_varlen(10 + hq + bs, [3, 1, 5, 2], [11, 9, 5, 0 + 2], hq=hq, hkv=hkv, d=8, bs=bs)
    kc, vc = _filled_pools(case)
    got = oracle.paged_attention_varlen(case.q, kc, vc, case.query_start_loc, case.seq_lens,
                                        case.block_tables, causal, case.scale)
    want = _brute_force_pool_scan(case, kc, vc, causal)
    assert torch.allclose(got, want, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- library special case

@pytest.mark.parametrize("hq,hkv", [(8, 2), (4, 4), (6, 3)])
def test_full_prefill_matches_torch_sdpa(hq, hkv):
    L, D, bs = 37, 16, 4
    case = _tiny_varlen(20 + hq, [L], [L], hq=hq, hkv=hkv, d=D, bs=bs)
    kc, vc = _filled_pools(case)
    got = oracle.paged_attention_varlen(case.q, kc, vc, case.query_start_loc, case.seq_lens,
                                        case.block_tables, True, case.scale)
    G = hq // hkv
    q = case.q.double().permute(1, 0, 2)[None]                               # [1, Hq, L, D]
    k = case.key.double().repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    v = case.value.double().repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    want = F.scaled_dot_product_attention(q, k, v, is_causal=True, scale=case.scale)[0].permute(1, 0, 2)
    assert torch.allclose(got, want, rtol=0, atol=1e-12)


def test_decode_matches_torch_sdpa():
    case = _tiny_varlen(30, [1, 1, 1], [19, 1, 40], hq=8, hkv=2, d=16, bs=4)
    kc, vc = _filled_pools(case)
    got = oracle.paged_attention_decode(case.q, kc, vc, case.block_tables, case.seq_lens, case.scale)
    off = 0
    for s, L in enumerate(case.seq_lens.tolist()):
        k = case.key[off:off + L].double().repeat_interleave(4, dim=1).permute(1, 0, 2)[None]
        v = case.value[off:off + L].double().repeat_interleave(4, dim=1).permute(1, 0, 2)[None]
        off += L
        q = case.q[s].double()[None, :, None, :]                              # [1, Hq, 1, D]
        want = F.scaled_dot_product_attention(q, k, v, scale=case.scale)[0, :, 0, :]
        assert torch.allclose(got[s], want, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- invariants

def test_page_permutation_invariance():
    a = _tiny_varlen(40, [2, 1], [14, 23], pool_extra=5)
    kc, vc = _filled_pools(a)
    out_a = oracle.paged_attention_varlen(a.q, kc, vc, a.query_start_loc, a.seq_lens, a.block_tables, True, a.scale)
    # same logical tokens, pages moved to other pool ids
    perm = torch.randperm(a.num_blocks, generator=torch.Generator().manual_seed(7)).to(torch.int32)
    tables = perm[a.block_tables.long()]
    kc2 = torch.full_like(kc, float("nan"))
    vc2 = torch.full_like(vc, float("nan"))
    kc2[perm.long()] = kc
    vc2[perm.long()] = vc
    out_b = oracle.paged_attention_varlen(a.q, kc2, vc2, a.query_start_loc, a.seq_lens, tables, True, a.scale)
    assert torch.equal(out_a, out_b)


def test_gqa_equals_repeated_kv_heads():
    case = _tiny_varlen(50, [4, 1], [17, 30], hq=8, hkv=2)
    kc, vc = _filled_pools(case)
    out = oracle.paged_attention_varlen(case.q, kc, vc, case.query_start_loc, case.seq_lens,
                                        case.block_tables, True, case.scale)
    kc_rep = kc.repeat_interleave(4, dim=2)
    vc_rep = vc.repeat_interleave(4, dim=2)
    out_rep = oracle.paged_attention_varlen(case.q, kc_rep, vc_rep, case.query_start_loc, case.seq_lens,
                                            case.block_tables, True, case.scale)
    assert torch.allclose(out, out_rep, rtol=0, atol=1e-15)


def test_chunked_prefill_equals_full_prefill():
    L, chunk = 29, 9
    full = _tiny_varlen(60, [L], [L])
    kc, vc = _filled_pools(full)
    out_full = oracle.paged_attention_varlen(full.q, kc, vc, full.query_start_loc, full.seq_lens,
                                             full.block_tables, True, full.scale)
    # the last `chunk` queries as a chunk over a context of L (prior L - chunk)
    qsl = torch.tensor([0, chunk], dtype=torch.int32)
    out_chunk = oracle.paged_attention_varlen(full.q[L - chunk:], kc, vc, qsl, full.seq_lens,
                                              full.block_tables, True, full.scale)
    assert torch.allclose(out_chunk, out_full[L - chunk:], rtol=0, atol=1e-14)


def test_varlen_qlen1_equals_decode():
    case = _tiny_varlen(70, [1, 1, 1], [5, 18, 33])
    kc, vc = _filled_pools(case)
    a = oracle.paged_attention_varlen(case.q, kc, vc, case.query_start_loc, case.seq_lens,
                                      case.block_tables, True, case.scale)
    b = oracle.paged_attention_decode(case.q, kc, vc, case.block_tables, case.seq_lens, case.scale)
    assert torch.allclose(a, b, rtol=0, atol=1e-15)


def test_token_subset_matches_full_evaluation():
    case = _tiny_varlen(80, [6, 2], [10, 7])
    kc, vc = _filled_pools(case)
    full = oracle.paged_attention_varlen(case.q, kc, vc, case.query_start_loc, case.seq_lens,
                                         case.block_tables, True, case.scale)
    subset = torch.tensor([1, 5, 7])
    part = oracle.paged_attention_varlen(case.q, kc, vc, case.query_start_loc, case.seq_lens,
                                         case.block_tables, True, case.scale, tokens=subset)
    # the library matmul may block a 3-row product differently from the full one
    assert torch.allclose(part[subset], full[subset], rtol=0, atol=1e-14)
    others = [i for i in range(case.num_tokens) if i not in subset.tolist()]
    assert torch.equal(part[others], torch.zeros_like(part[others]))


def test_default_scale():
    assert oracle.default_scale(128, 0.0) == 1.0 / math.sqrt(128)
    assert oracle.default_scale(64, None) == 0.125
    assert oracle.default_scale(64, 0.3) == 0.3


def test_rejects_query_longer_than_context():
    case = _tiny_varlen(90, [3], [3])
    kc, vc = _filled_pools(case)
    with pytest.raises(ValueError):
        oracle.paged_attention_varlen(case.q, kc, vc, case.query_start_loc,
                                      torch.tensor([2], dtype=torch.int32), case.block_tables, True)


# --------------------------------------------------------------------------- reshape_and_cache

def test_reshape_and_cache_golden():
    g = _load("reshape_and_cache_tiny.json")
    shape = (g["num_blocks"], g["block_size"], g["num_kv_heads"], g["head_dim"])
    kc = torch.full(shape, g["fill"], dtype=torch.float32)
    vc = torch.full(shape, g["fill"], dtype=torch.float32)
    oracle.reshape_and_cache(torch.tensor(g["key"], dtype=torch.float32),
                             torch.tensor(g["value"], dtype=torch.float32), kc, vc,
                             torch.tensor(g["slot_mapping"], dtype=torch.int32))
    assert torch.equal(kc, torch.tensor(g["expected_k_cache"], dtype=torch.float32))
    assert torch.equal(vc, torch.tensor(g["expected_v_cache"], dtype=torch.float32))


def test_reshape_and_cache_round_trip_through_gather():
    case = _tiny_varlen(100, [1, 1, 1], [13, 4, 21], dtype=torch.bfloat16)
    kc, vc = _filled_pools(case)
    off = 0
    for r, L in enumerate(case.seq_lens.tolist()):
        assert torch.equal(oracle.gather_context(kc, case.block_tables[r], L),
                           case.key[off:off + L].double())
        assert torch.equal(oracle.gather_context(vc, case.block_tables[r], L),
                           case.value[off:off + L].double())
        off += L


def test_reshape_and_cache_rejects_slot_outside_pool():
    kc = torch.zeros((2, 4, 1, 8))
    vc = torch.zeros((2, 4, 1, 8))
    with pytest.raises(ValueError):
        oracle.reshape_and_cache(torch.ones((1, 1, 8)), torch.ones((1, 1, 8)), kc, vc,
                                 torch.tensor([8], dtype=torch.int32))
