"""Pins for the cascade (shared-prefix) oracle: with a page-aligned prefix it is a plain decode
over the concatenated block table; an empty prefix is a plain decode over the suffix; an empty
suffix is the prefix alone; and it matches torch SDPA over the concatenated keys."""

import torch
import torch.nn.functional as F

import oracle
import workloads


def _setup(prefix_len, suffix_lens, bs=4, hq=4, hkv=2, d=8, seed=0):
    # one case holding the prefix (request 0) and the suffixes (requests 1..S)
    case = workloads.make_case("c", seed, [1] * (1 + len(suffix_lens)), [prefix_len] + suffix_lens,
                               num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs, dtype=torch.float64,
                               table_multiple=4, pool_blocks=sum(workloads.cdiv(L, bs) for L in
                                                                 [prefix_len] + suffix_lens) + 2)
    kc, vc = case.empty_pools()
    oracle.reshape_and_cache(case.key, case.value, kc, vc, case.slot_mapping)
    q = case.q[1:]
    return case, kc, vc, q


def test_page_aligned_prefix_equals_plain_decode():
    bs, P = 4, 12
    case, kc, vc, q = _setup(P, [5, 9, 1], bs=bs)
    out = oracle.cascade_decode(q, kc, vc, case.block_tables[0], P, case.block_tables[1:], case.seq_lens[1:],
                                case.scale)
    n_pre = P // bs
    tables = torch.cat([case.block_tables[0, :n_pre].expand(3, -1), case.block_tables[1:]], dim=1)
    lens = case.seq_lens[1:] + P
    want = oracle.paged_attention_decode(q, kc, vc, tables, lens, case.scale)
    assert torch.allclose(out, want, rtol=0, atol=1e-15)


def test_empty_prefix_or_suffix():
    case, kc, vc, q = _setup(10, [7, 3])
    empty = oracle.cascade_decode(q, kc, vc, case.block_tables[0], 0, case.block_tables[1:], case.seq_lens[1:],
                                  case.scale)
    plain = oracle.paged_attention_decode(q, kc, vc, case.block_tables[1:], case.seq_lens[1:], case.scale)
    assert torch.equal(empty, plain)
    no_suffix = oracle.cascade_decode(q, kc, vc, case.block_tables[0], 10, case.block_tables[1:],
                                      torch.zeros(2, dtype=torch.int32), case.scale)
    prefix_only = oracle.paged_attention_decode(q, kc, vc, case.block_tables[0:1].expand(2, -1),
                                                torch.tensor([10, 10], dtype=torch.int32), case.scale)
    assert torch.allclose(no_suffix, prefix_only, rtol=0, atol=1e-15)


def test_matches_sdpa_over_concatenated_keys():
    P, suffix = 11, [6, 13]
    case, kc, vc, q = _setup(P, suffix, hq=4, hkv=4, seed=3)
    out = oracle.cascade_decode(q, kc, vc, case.block_tables[0], P, case.block_tables[1:], case.seq_lens[1:],
                                case.scale)
    off = [0, P, P + suffix[0]]
    for s in range(2):
        k = torch.cat([case.key[:P], case.key[off[s + 1]:off[s + 1] + suffix[s]]]).double().permute(1, 0, 2)[None]
        v = torch.cat([case.value[:P], case.value[off[s + 1]:off[s + 1] + suffix[s]]]).double().permute(1, 0, 2)[None]
        want = F.scaled_dot_product_attention(q[s].double()[None, :, None, :], k, v, scale=case.scale)[0, :, 0]
        assert torch.allclose(out[s], want, rtol=0, atol=1e-12)
