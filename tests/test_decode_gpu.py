"""GPU parity of the split-KV decode (pa_paged_attention_decode) against the float64 oracle."""

import pytest
import torch

import oracle
import paged_kv_attention_gb300 as pa
import workloads
from paged_helpers import check_close, gpu_pools, named_case, oracle_pools

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_decode(case, kc, vc, splits=0, **kw):
    return pa.paged_attention_decode(case.q.to(DEV), kc, vc, case.block_tables.to(DEV),
                                     case.seq_lens.to(DEV), case.scale, num_splits=splits, **kw)


def oracle_decode(case, ko, vo):
    return oracle.paged_attention_decode(case.q, ko, vo, case.block_tables, case.seq_lens, case.scale)


@pytest.mark.parametrize("name", ["decode_1seq_fp32", "decode_ragged32_bf16", "decode_64x4096_bf16",
                                  "decode_64x4096_bf16_d256"])
def test_named_workloads(name):
    case, (ko, vo) = named_case(name)
    kc, vc = gpu_pools(case)
    out = run_decode(case, kc, vc)
    check_close(out, oracle_decode(case, ko, vo), case.dtype, label=name)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("splits", [1, 3, 8, 0])
def test_split_counts(dtype, splits):
    case = workloads.decode_case("splits", 11, [1, 600, 1500, 17, 4096, 0, 333], num_q_heads=32,
                                 num_kv_heads=8, head_dim=128, block_size=16, dtype=dtype, pool_blocks=600)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    out = run_decode(case, kc, vc, splits)
    check_close(out, oracle_decode(case, ko, vo), dtype, label=f"splits={splits}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("head_dim", [64, 128, 256])
@pytest.mark.parametrize("splits", [17, 20, 32])
def test_many_splits(dtype, head_dim, splits):
    """More than 16 splits: the combine's per-split weights come from lanes 16-31 too."""
    hq, hkv = (16, 4) if dtype == torch.bfloat16 or head_dim < 256 else (8, 4)
    case = workloads.decode_case("many", 150 + head_dim + splits, [1, 333, 1500, 4096], num_q_heads=hq,
                                 num_kv_heads=hkv, head_dim=head_dim, block_size=16, dtype=dtype)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    out = run_decode(case, kc, vc, splits)
    check_close(out, oracle_decode(case, ko, vo), dtype, label=f"D{head_dim} splits={splits}")


@pytest.mark.parametrize("head_dim", [64, 128, 256])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (12, 4), (16, 4), (32, 4), (32, 2)])
@pytest.mark.parametrize("block_size", [16, 32, 64])
def test_shapes_bf16(head_dim, hq, hkv, block_size):
    lens = [1, 15, 16, 17, 130, 777]
    case = workloads.decode_case("shapes", 100 + head_dim + hq + block_size, lens, num_q_heads=hq,
                                 num_kv_heads=hkv, head_dim=head_dim, block_size=block_size,
                                 dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    for splits in (1, 4):
        out = run_decode(case, kc, vc, splits)
        check_close(out, oracle_decode(case, ko, vo), torch.bfloat16, label=f"D{head_dim} G{hq // hkv} bs{block_size}")


@pytest.mark.parametrize("head_dim,hq,hkv", [(64, 8, 2), (128, 8, 8), (128, 24, 8), (256, 16, 2), (128, 32, 2)])
@pytest.mark.parametrize("block_size", [1, 8, 16])
def test_shapes_fp32(head_dim, hq, hkv, block_size):
    lens = [3, 31, 32, 33, 200]
    case = workloads.decode_case("f32", 200 + head_dim + block_size, lens, num_q_heads=hq, num_kv_heads=hkv,
                                 head_dim=head_dim, block_size=block_size, dtype=torch.float32)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    for splits in (1, 2):
        out = run_decode(case, kc, vc, splits)
        check_close(out, oracle_decode(case, ko, vo), torch.float32, label=f"f32 D{head_dim} bs{block_size}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_page_permutation_is_bitwise_invariant(dtype):
    """Moving pages to other pool ids changes addresses, not arithmetic (fixed split count)."""
    a = workloads.decode_case("perm", 21, [70, 513, 1000], num_q_heads=16, num_kv_heads=4, head_dim=128,
                              block_size=16, dtype=dtype, pool_blocks=200)
    b = workloads.decode_case("perm", 22, [70, 513, 1000], num_q_heads=16, num_kv_heads=4, head_dim=128,
                              block_size=16, dtype=dtype, pool_blocks=200)
    b.q, b.key, b.value = a.q, a.key, a.value          # same logical data, other page ids
    assert not torch.equal(a.block_tables, b.block_tables)
    kca, vca = gpu_pools(a)
    kcb, vcb = gpu_pools(b)
    oa = run_decode(a, kca, vca, 3)
    ob = run_decode(b, kcb, vcb, 3)
    assert torch.equal(oa, ob)


def test_poisoned_memory_never_leaks():
    """Pools are NaN outside the written slots (tails of last pages, unused pages, padding
    table entries); every output must stay finite, including zero-length rows."""
    case = workloads.decode_case("poison", 31, [0, 1, 5, 16, 17, 31, 1000], num_q_heads=32, num_kv_heads=8,
                                 head_dim=128, block_size=16, dtype=torch.bfloat16, pool_blocks=150)
    kc, vc = gpu_pools(case)
    for splits in (1, 5, 0):
        out = run_decode(case, kc, vc, splits)
        assert torch.isfinite(out.float()).all()
        assert torch.equal(out[0], torch.zeros_like(out[0]))


def test_cuda_graph_replay_follows_device_lengths():
    """Launch shape depends on host sizes only: a captured decode replays correctly after the
    lengths (device buffer) grow and new tokens are written."""
    S, full = 4, [300, 900, 64, 1200]
    case = workloads.decode_case("graph", 41, full, num_q_heads=32, num_kv_heads=8, head_dim=128,
                                 block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    q = case.q.to(DEV)
    tables = case.block_tables.to(DEV)
    lens = torch.tensor([200, 700, 10, 1100], dtype=torch.int32, device=DEV)
    out = torch.empty_like(q)
    ws = torch.empty(pa.decode_workspace_bytes(S, 32, 128, tables.shape[1], 16, 0), dtype=torch.uint8, device=DEV)
    pa.paged_attention_decode(q, kc, vc, tables, lens, case.scale, out=out, workspace=ws)  # warm-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pa.paged_attention_decode(q, kc, vc, tables, lens, case.scale, out=out, workspace=ws)
    ko, vo = oracle_pools(case)
    for step in range(3):
        new = torch.tensor([200 + 50 * step, 700 + 100 * step, 10 + 27 * step, 1100 + 33 * step], dtype=torch.int32)
        lens.copy_(new.to(DEV))
        g.replay()
        torch.cuda.synchronize()
        eager = pa.paged_attention_decode(q, kc, vc, tables, lens, case.scale, workspace=ws)
        assert torch.equal(out, eager)
        want = oracle.paged_attention_decode(case.q, ko, vo, case.block_tables, new, case.scale)
        check_close(out, want, torch.bfloat16, label=f"graph step {step}")


def test_error_word_flags_bad_pages_and_lengths():
    case = workloads.decode_case("err", 51, [40, 40, 40], num_q_heads=8, num_kv_heads=2, head_dim=128,
                                 block_size=16, dtype=torch.bfloat16, pool_blocks=12)
    kc, vc = gpu_pools(case)
    for dtype_case in (case,):
        tables = dtype_case.block_tables.clone()
        tables[1, 1] = 10_000                      # page id outside the pool
        lens = dtype_case.seq_lens.clone()
        lens[2] = tables.shape[1] * 16 + 5         # longer than the table can hold
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = pa.paged_attention_decode(case.q.to(DEV), kc, vc, tables.to(DEV), lens.to(DEV), case.scale,
                                        num_splits=1, error_word=err)
        torch.cuda.synchronize()
        bits = int(err.item())
        assert bits & pa._lib.PA_ERRBIT_PAGE_OUT_OF_POOL
        assert bits & pa._lib.PA_ERRBIT_LENGTH_OUT_OF_RANGE
        # the untouched sequence is still right
        ko, vo = oracle_pools(case)
        want = oracle.paged_attention_decode(case.q, ko, vo, case.block_tables, case.seq_lens, case.scale)
        check_close(out[0:1], want[0:1], torch.bfloat16, label="clean row")


def test_workspace_too_small_is_refused():
    case = workloads.decode_case("ws", 61, [2000, 2000], num_q_heads=8, num_kv_heads=2, head_dim=128,
                                 block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    small = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(pa.PagedAttentionError) as e:
        run_decode(case, kc, vc, 8, workspace=small)
    assert e.value.status == pa._lib.PA_ERR_WORKSPACE_TOO_SMALL
