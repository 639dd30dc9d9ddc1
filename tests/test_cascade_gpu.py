"""GPU parity of the cascade (shared-prefix) decode, pa_cascade_decode, against the float64
oracle's cascade_decode: the prefix pass on the tensor cores, the suffix split-KV decode and the
log-sum-exp combine together."""

import pytest
import torch

import oracle
import paged_kv_attention_gb300 as pa
import workloads
from paged_helpers import check_close, gpu_pools, named_case, oracle_pools

pytestmark = pytest.mark.gpu
DEV = "cuda"


def suffix_tables(case):
    """The suffix rows of the case's block table, trimmed to the widest suffix's pages."""
    width = max(1, workloads.cdiv(int(case.seq_lens[1:].max()), case.block_size))
    return case.block_tables[1:, :width].contiguous()


def run_cascade(case, kc, vc, prefix_len=None, splits=0, **kw):
    plen = int(case.seq_lens[0]) if prefix_len is None else prefix_len
    return pa.cascade_decode(case.q.to(DEV), kc, vc, case.block_tables[0].to(DEV),
                             torch.tensor([plen], dtype=torch.int32, device=DEV), suffix_tables(case).to(DEV),
                             case.seq_lens[1:].to(DEV), case.scale, num_splits=splits, **kw)


def oracle_cascade(case, ko, vo, prefix_len=None):
    plen = int(case.seq_lens[0]) if prefix_len is None else prefix_len
    return oracle.cascade_decode(case.q, ko, vo, case.block_tables[0], plen, case.block_tables[1:],
                                 case.seq_lens[1:], case.scale)


def test_named_64_sequences_sharing_4000_tokens():
    case, (ko, vo) = named_case("cascade_64x4000_bf16")
    kc, vc = gpu_pools(case)
    out = run_cascade(case, kc, vc)
    check_close(out, oracle_cascade(case, ko, vo), torch.bfloat16, label="cascade 64x4000")


@pytest.mark.parametrize("prefix_len", [0, 1, 37, 128, 129, 1000, 2050])
@pytest.mark.parametrize("hq,hkv,bs", [(32, 8, 16), (8, 8, 16), (16, 2, 64), (16, 1, 32), (4, 2, 128)])
def test_prefix_lengths_and_groups(prefix_len, hq, hkv, bs):
    suffix = [0, 1, 5, 16, 17, 200, 333]
    case = workloads.cascade_case("cs", 500 + prefix_len + hq + bs, prefix_len, suffix, num_q_heads=hq,
                                  num_kv_heads=hkv, head_dim=128, block_size=bs, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    want = oracle_cascade(case, ko, vo)
    for splits in (1, 3, 0):
        out = run_cascade(case, kc, vc, splits=splits)
        # a sequence with an empty prefix and an empty suffix has no keys: zeros
        if prefix_len == 0:
            assert torch.equal(out[0].float(), torch.zeros_like(out[0].float()))
        check_close(out, want, torch.bfloat16, label=f"P{prefix_len} G{hq // hkv} bs{bs} splits={splits}")


@pytest.mark.parametrize("prefix_len", [0, 37, 1000])
@pytest.mark.parametrize("hq,hkv,bs", [(32, 8, 16), (16, 1, 32), (8, 4, 64)])
def test_head_dim_64(prefix_len, hq, hkv, bs):
    """The prefix pass at head_dim 64 (one 64-column block per row), several suffix splits."""
    suffix = [0, 1, 17, 200, 333, 64]
    case = workloads.cascade_case("c64", 900 + prefix_len + hq + bs, prefix_len, suffix, num_q_heads=hq,
                                  num_kv_heads=hkv, head_dim=64, block_size=bs, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    want = oracle_cascade(case, ko, vo)
    for splits in (1, 0):
        out = run_cascade(case, kc, vc, splits=splits)
        check_close(out, want, torch.bfloat16, label=f"D64 P{prefix_len} G{hq // hkv} bs{bs} splits={splits}")


@pytest.mark.parametrize("num_seqs", [1, 63, 64, 65, 130, 300])
def test_many_sequences_span_query_tiles(num_seqs):
    """More sequences than one CTA's query rows (64 at G=4): several prefix tiles, ragged last."""
    gen = torch.Generator().manual_seed(700 + num_seqs)
    suffix = torch.randint(0, 300, (num_seqs,), generator=gen).tolist()
    case = workloads.cascade_case("cn", 700 + num_seqs, 777, suffix, num_q_heads=32, num_kv_heads=8, head_dim=128,
                                  block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    out = run_cascade(case, kc, vc)
    check_close(out, oracle_cascade(case, ko, vo), torch.bfloat16, label=f"S={num_seqs}")


def test_matches_plain_decode_over_concatenated_tables():
    """A page-aligned prefix makes the cascade a plain decode over [prefix pages, suffix pages]."""
    P, bs = 1024, 16
    suffix = [3, 90, 250, 17]
    case = workloads.cascade_case("cp", 801, P, suffix, num_q_heads=32, num_kv_heads=8, head_dim=128,
                                  block_size=bs, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    out = run_cascade(case, kc, vc)
    n_pre = P // bs
    tables = torch.cat([case.block_tables[0, :n_pre].expand(len(suffix), -1), suffix_tables(case)], dim=1)
    plain = pa.paged_attention_decode(case.q.to(DEV), kc, vc, tables.contiguous().to(DEV),
                                      (case.seq_lens[1:] + P).to(DEV), case.scale)
    diff = (out.float() - plain.float()).abs()
    assert diff.max().item() <= 2e-2 and diff.mean().item() <= 2e-3


def test_cuda_graph_replay_follows_device_lengths():
    """prefix_len and suffix_lens are device values: a captured cascade follows both growing."""
    case = workloads.cascade_case("cg", 811, 1500, [400, 10, 250], num_q_heads=32, num_kv_heads=8, head_dim=128,
                                  block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    q = case.q.to(DEV)
    ptable = case.block_tables[0].to(DEV)
    stables = suffix_tables(case).to(DEV)
    plen = torch.tensor([900], dtype=torch.int32, device=DEV)
    slens = torch.tensor([100, 1, 50], dtype=torch.int32, device=DEV)
    out = torch.empty_like(q)
    ws = torch.empty(pa._lib.load().pa_cascade_workspace_bytes(3, 32, 128, 16, ptable.numel(), stables.shape[1]),
                     dtype=torch.uint8, device=DEV)
    pa.cascade_decode(q, kc, vc, ptable, plen, stables, slens, case.scale, out=out, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pa.cascade_decode(q, kc, vc, ptable, plen, stables, slens, case.scale, out=out, workspace=ws)
    for step in range(3):
        p_now = 900 + 250 * step
        s_now = torch.tensor([100 + 120 * step, 1 + 4 * step, 50 + 90 * step], dtype=torch.int32)
        plen.fill_(p_now)
        slens.copy_(s_now.to(DEV))
        g.replay()
        torch.cuda.synchronize()
        want = oracle.cascade_decode(case.q, ko, vo, case.block_tables[0], p_now, case.block_tables[1:], s_now,
                                     case.scale)
        check_close(out, want, torch.bfloat16, label=f"cascade graph step {step}")


def test_prefix_length_out_of_range_is_flagged():
    case = workloads.cascade_case("cf", 821, 40, [5, 6], num_q_heads=8, num_kv_heads=2, head_dim=128,
                                  block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    cap = case.block_tables.shape[1] * 16
    run_cascade(case, kc, vc, prefix_len=cap + 3, error_word=err)   # clamped to the table's capacity
    torch.cuda.synchronize()
    assert int(err.item()) & pa._lib.PA_ERRBIT_LENGTH_OUT_OF_RANGE
    err.zero_()
    run_cascade(case, kc, vc, prefix_len=-1, error_word=err)        # clamped to an empty prefix
    torch.cuda.synchronize()
    assert int(err.item()) & pa._lib.PA_ERRBIT_LENGTH_OUT_OF_RANGE


def test_workspace_too_small_and_unsupported_shapes():
    case = workloads.cascade_case("cw", 831, 300, [20, 30], num_q_heads=8, num_kv_heads=2, head_dim=128,
                                  block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    with pytest.raises(pa.PagedAttentionError) as e:
        run_cascade(case, kc, vc, workspace=torch.empty(16, dtype=torch.uint8, device=DEV))
    assert e.value.status == pa._lib.PA_ERR_WORKSPACE_TOO_SMALL
    small = workloads.cascade_case("cu", 832, 300, [20, 30], num_q_heads=8, num_kv_heads=2, head_dim=256,
                                   block_size=16, dtype=torch.bfloat16)
    kc2, vc2 = gpu_pools(small)
    with pytest.raises(pa.PagedAttentionError) as e:
        run_cascade(small, kc2, vc2)
    assert e.value.status == pa._lib.PA_ERR_UNSUPPORTED
