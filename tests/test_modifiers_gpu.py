"""GPU parity of the score modifiers (sliding window, logit softcap, attention sinks) on every
path: split-KV decode (bf16 and fp32, several split counts), the tcgen05 varlen kernel
(head_dim 128) and the generic varlen path (head_dim 64)."""

import pytest
import torch

import oracle
import paged_kv_attention_gb300 as pa
import workloads
from paged_helpers import check_close, gpu_pools, oracle_pools

pytestmark = pytest.mark.gpu
DEV = "cuda"

MODS = [dict(window=1), dict(window=37), dict(window=300), dict(window=5000), dict(softcap=5.0),
        dict(sinks=True), dict(window=100, softcap=3.0, sinks=True)]


def _sinks(hq, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(hq, generator=g, dtype=torch.float32) * 2.0)


def _kw(mod, hq, seed):
    kw = dict(window=mod.get("window", 0), softcap=mod.get("softcap", 0.0))
    sinks = _sinks(hq, seed) if mod.get("sinks") else None
    return kw, sinks


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("splits", [1, 4, 0])
@pytest.mark.parametrize("mod", MODS, ids=lambda m: "-".join(f"{k}{v}" for k, v in m.items()))
def test_decode_modifiers(dtype, splits, mod):
    case = workloads.decode_case("dmod", 901, [1, 40, 333, 1500, 17], num_q_heads=16, num_kv_heads=4,
                                 head_dim=128 if dtype == torch.bfloat16 else 64, block_size=16, dtype=dtype)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    kw, sinks = _kw(mod, case.num_q_heads, 7)
    out = pa.paged_attention_decode(case.q.to(DEV), kc, vc, case.block_tables.to(DEV), case.seq_lens.to(DEV),
                                    case.scale, num_splits=splits, sinks=None if sinks is None else sinks.to(DEV),
                                    **kw)
    want = oracle.paged_attention_decode(case.q, ko, vo, case.block_tables, case.seq_lens, case.scale,
                                         sinks=None if sinks is None else sinks.double(), **kw)
    check_close(out, want, dtype, label=f"decode {mod} splits={splits}")


@pytest.mark.parametrize("head_dim,hq,hkv,bs,dtype", [(128, 32, 8, 16, torch.bfloat16),   # tcgen05 kernel
                                                      (128, 16, 16, 64, torch.bfloat16),  # tcgen05, G = 1
                                                      (64, 16, 4, 16, torch.bfloat16),    # generic path
                                                      (64, 8, 2, 16, torch.float32)])     # generic, fp32
@pytest.mark.parametrize("mod", MODS, ids=lambda m: "-".join(f"{k}{v}" for k, v in m.items()))
def test_varlen_modifiers(head_dim, hq, hkv, bs, dtype, mod):
    q_lens = [300, 1, 5, 64, 0, 129]
    seq_lens = [700, 900, 33, 64, 8, 1500]
    case = workloads.make_case("vmod", 902 + head_dim + hq, q_lens, seq_lens, num_q_heads=hq, num_kv_heads=hkv,
                               head_dim=head_dim, block_size=bs, dtype=dtype)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    kw, sinks = _kw(mod, hq, 11)
    out = pa.paged_attention_varlen(case.q.to(DEV), kc, vc, case.query_start_loc.to(DEV), case.seq_lens.to(DEV),
                                    case.block_tables.to(DEV), case.max_query_len, True, case.scale,
                                    sinks=None if sinks is None else sinks.to(DEV), **kw)
    want = oracle.paged_attention_varlen(case.q, ko, vo, case.query_start_loc, case.seq_lens, case.block_tables,
                                         True, case.scale, sinks=None if sinks is None else sinks.double(), **kw)
    check_close(out, want, dtype, label=f"varlen D{head_dim} G{hq // hkv} {mod}")


def test_long_prefill_with_window_skips_old_tiles():
    """A 4096-token prompt with a 700-key window: most CTAs start several key tiles in."""
    L, w = 4096, 700
    case = workloads.make_case("pw", 903, [L], [L], num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=64,
                               dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    out = pa.paged_attention_varlen(case.q.to(DEV), kc, vc, case.query_start_loc.to(DEV), case.seq_lens.to(DEV),
                                    case.block_tables.to(DEV), L, True, case.scale, window=w)
    rows = torch.cat([torch.arange(0, 200), torch.arange(650, 800), torch.arange(L - 300, L), torch.arange(0, L, 97)])
    rows = torch.unique(rows)
    want = oracle.paged_attention_varlen(case.q, ko, vo, case.query_start_loc, case.seq_lens, case.block_tables,
                                         True, case.scale, tokens=rows, window=w)
    check_close(out, want, torch.bfloat16, rows=rows, label="prefill window")


def test_bad_options_are_refused():
    case = workloads.decode_case("opt", 904, [10], num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                                 dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    for kw in (dict(window=-1), dict(softcap=-2.0), dict(softcap=float("inf"))):
        with pytest.raises(pa.PagedAttentionError) as e:
            pa.paged_attention_decode(case.q.to(DEV), kc, vc, case.block_tables.to(DEV), case.seq_lens.to(DEV),
                                      case.scale, **kw)
        assert e.value.status == pa._lib.PA_ERR_INVALID_ARGUMENT
