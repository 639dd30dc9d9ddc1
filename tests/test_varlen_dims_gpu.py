"""GPU parity of the tensor-core varlen kernels at head_dim 64 and 256 against the float64 oracle:
mixed batches of prefill chunks, decodes and verify blocks over every supported GQA group and
block size, causal and not, with score modifiers, on the default, planned and split grids, a long
prompt, CUDA-graph replay and invariances. At 64 a CTA's two query tiles share each K/V tile; at
256 it runs them one after the other, its scores double-buffered in tensor memory and its K/V in a
ring of half tiles ("32. Production attention kernels", One kernel for the whole batch)."""

import pytest
import torch

import oracle
import paged_kv_attention_gb300 as pa
import workloads
from paged_helpers import check_close, gpu_pools, oracle_pools

pytestmark = pytest.mark.gpu
DEV = "cuda"

Q_LENS = [37, 1, 5, 0, 130, 300, 64, 1, 129]
SEQ_LENS = [90, 700, 2000, 3, 900, 300, 1000, 17, 129]


def run(case, kc, vc, causal=None, **kw):
    return pa.paged_attention_varlen(case.q.to(DEV), kc, vc, case.query_start_loc.to(DEV), case.seq_lens.to(DEV),
                                     case.block_tables.to(DEV), case.max_query_len,
                                     case.causal if causal is None else causal, case.scale, **kw)


def want(case, ko, vo, causal=None, **kw):
    return oracle.paged_attention_varlen(case.q, ko, vo, case.query_start_loc, case.seq_lens, case.block_tables,
                                         case.causal if causal is None else causal, case.scale, **kw)


@pytest.mark.parametrize("head_dim", [64, 256])
@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("bs", [16, 32, 64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_mixed_batches(head_dim, G, bs, causal):
    hkv = 2 if G <= 8 else 1
    case = workloads.make_case("vdim", 2000 + head_dim + 10 * G + bs, Q_LENS, SEQ_LENS, num_q_heads=G * hkv,
                               num_kv_heads=hkv, head_dim=head_dim, block_size=bs, dtype=torch.bfloat16,
                               causal=causal)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    check_close(run(case, kc, vc), want(case, ko, vo), torch.bfloat16,
                label=f"D{head_dim} G{G} bs{bs} causal={causal}")


@pytest.mark.parametrize("head_dim", [64, 256])
@pytest.mark.parametrize("window,softcap,sinks", [(100, 0.0, False), (0, 30.0, False), (0, 0.0, True),
                                                  (37, 20.0, True), (700, 0.0, False)])
def test_score_modifiers(head_dim, window, softcap, sinks):
    hq, hkv = (32, 8) if head_dim == 64 else (16, 4)
    case = workloads.make_case("vdimm", 2100 + head_dim + window, Q_LENS, SEQ_LENS, num_q_heads=hq,
                               num_kv_heads=hkv, head_dim=head_dim, block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    sk = torch.linspace(-2.0, 3.0, hq, dtype=torch.float32) if sinks else None
    out = run(case, kc, vc, window=window, softcap=softcap, sinks=None if sk is None else sk.to(DEV))
    check_close(out, want(case, ko, vo, window=window, softcap=softcap, sinks=sk), torch.bfloat16,
                label=f"D{head_dim} w{window} cap{softcap} sinks{sinks}")


@pytest.mark.parametrize("head_dim", [64, 256])
@pytest.mark.parametrize("split", [False, True])
def test_planned_grid_and_split_path(head_dim, split):
    """The planned grid gives the default grid's result bit for bit; the split path (short
    requests on the split-KV decode) agrees with the oracle."""
    hq, hkv = (32, 8) if head_dim == 64 else (16, 4)
    case = workloads.make_case("vdimp", 2200 + head_dim, Q_LENS, SEQ_LENS, num_q_heads=hq, num_kv_heads=hkv,
                               head_dim=head_dim, block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    base = run(case, kc, vc, split_decodes=split)
    items = pa.varlen_plan(case.query_start_loc, case.seq_lens, case.max_query_len, hq, hkv, True, 0,
                           split_decodes=split)
    planned = run(case, kc, vc, split_decodes=split, work_items=items.to(DEV))
    assert torch.equal(base, planned)
    check_close(base, want(case, ko, vo), torch.bfloat16, label=f"D{head_dim} split={split}")


@pytest.mark.parametrize("head_dim,hq,hkv,bs", [(256, 16, 4, 64), (256, 8, 1, 16), (64, 32, 8, 64)])
def test_long_prompt_every_row(head_dim, hq, hkv, bs):
    """One 3,000-token causal prompt (a ragged last tile pair) plus a 1,000-token chunk after 2,000
    cached positions: every row against the oracle."""
    case = workloads.make_case("vdiml", 2300 + head_dim + bs, [3000, 1000], [3000, 3000], num_q_heads=hq,
                               num_kv_heads=hkv, head_dim=head_dim, block_size=bs, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    check_close(run(case, kc, vc), want(case, ko, vo), torch.bfloat16, label=f"long D{head_dim} G{hq // hkv}")


@pytest.mark.parametrize("head_dim", [64, 256])
def test_page_permutation_is_bitwise_invariant(head_dim):
    """The same logical context on a differently permuted pool gives the same bits: the pages only
    move where the copies come from."""
    hq, hkv = (16, 4)
    a = workloads.make_case("vperm", 2400, [200, 33], [900, 500], num_q_heads=hq, num_kv_heads=hkv,
                            head_dim=head_dim, block_size=16, dtype=torch.bfloat16, pool_blocks=120)
    b = workloads.make_case("vperm", 2400, [200, 33], [900, 500], num_q_heads=hq, num_kv_heads=hkv,
                            head_dim=head_dim, block_size=16, dtype=torch.bfloat16, pool_blocks=120,
                            gen=torch.Generator().manual_seed(2401))
    b.q, b.key, b.value = a.q, a.key, a.value
    ka, va = gpu_pools(a)
    kb, vb = gpu_pools(b)
    assert not torch.equal(a.block_tables, b.block_tables)
    assert torch.equal(run(a, ka, va), run(b, kb, vb))


@pytest.mark.parametrize("head_dim", [64, 256])
def test_cuda_graph_replay_follows_device_positions(head_dim):
    hq, hkv = (16, 4)
    full = [700, 300, 1200]
    q_lens = [64, 1, 5]
    case = workloads.make_case("vdimg", 2500 + head_dim, q_lens, full, num_q_heads=hq, num_kv_heads=hkv,
                               head_dim=head_dim, block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    q = case.q.to(DEV)
    qsl = case.query_start_loc.to(DEV)
    tables = case.block_tables.to(DEV)
    lens = torch.tensor([500, 100, 900], dtype=torch.int32, device=DEV)
    out = torch.empty_like(q)
    pa.paged_attention_varlen(q, kc, vc, qsl, lens, tables, 64, True, case.scale, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pa.paged_attention_varlen(q, kc, vc, qsl, lens, tables, 64, True, case.scale, out=out)
    for step in range(3):
        new = torch.tensor([500 + 64 * step, 100 + 90 * step, 900 + 140 * step], dtype=torch.int32)
        lens.copy_(new.to(DEV))
        g.replay()
        torch.cuda.synchronize()
        w = oracle.paged_attention_varlen(case.q, ko, vo, case.query_start_loc, new, case.block_tables, True,
                                          case.scale)
        check_close(out, w, torch.bfloat16, label=f"D{head_dim} graph step {step}")


@pytest.mark.parametrize("head_dim", [64, 256])
def test_bad_request_is_flagged_and_zeroed(head_dim):
    case = workloads.make_case("vdimb", 2600 + head_dim, [4, 3], [10, 20], num_q_heads=8, num_kv_heads=2,
                               head_dim=head_dim, block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    bad_lens = case.seq_lens.clone()
    bad_lens[0] = 2
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pa.paged_attention_varlen(case.q.to(DEV), kc, vc, case.query_start_loc.to(DEV), bad_lens.to(DEV),
                                    case.block_tables.to(DEV), case.max_query_len, True, case.scale,
                                    error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa._lib.PA_ERRBIT_QUERY_LAYOUT
    assert torch.equal(out[:4].float(), torch.zeros_like(out[:4].float()))
    ko, vo = oracle_pools(case)
    check_close(out[4:], want(case, ko, vo)[4:], torch.bfloat16, label="clean request")
