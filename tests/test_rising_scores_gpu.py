"""GPU parity of the online softmax when a row's scores jump between key tiles.

Random keys give scores whose maximum is reached in the first key tile to within a few units,
so the running reference of the softmax almost never moves. Here every key of 128-key tile i
gets the same offset level[i] * (1, ..., 1) added, so that a query row's scores shift by
level[i] * z between tiles (z = scale * sum(q) ~ N(0, 1), either sign): rises of 8-64 octaves
and of more than 64 octaves (the reference moves and the accumulated output and row sum are
rescaled), and falls (the reference stays). Sinks far below or above the scores make the first
tile itself such a jump. The oracle follows the textbook softmax in float64."""

import pytest
import torch

import oracle
import paged_kv_attention_gb300 as pa
import workloads
from paged_helpers import check_close, gpu_pools, oracle_pools

DEV = "cuda"

LEVELS = [0.0, 10.0, 60.0, 0.0, 120.0, 125.0, -30.0, 126.0]


def rising_case(seed, q_lens, seq_lens, hq, hkv, bs, head_dim=128):
    case = workloads.make_case("rise", seed, q_lens, seq_lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=head_dim,
                               block_size=bs, dtype=torch.bfloat16)
    key = case.key.float()
    off = 0
    for L in seq_lens:
        tile = torch.arange(L) // 128
        lev = torch.tensor(LEVELS)[tile.clamp(max=len(LEVELS) - 1)]
        key[off:off + L] = key[off:off + L] * 0.5 + lev[:, None, None]
        off += L
    case.key = key.to(torch.bfloat16)
    return case


MODS = [dict(), dict(softcap=20.0), dict(window=200), dict(sinks=-100.0), dict(sinks=-40.0), dict(sinks=30.0),
        dict(window=300, softcap=30.0, sinks=-60.0)]


@pytest.mark.gpu
@pytest.mark.parametrize("hq,hkv,bs", [(32, 8, 16), (16, 16, 64), (16, 2, 32)])
@pytest.mark.parametrize("mod", MODS, ids=lambda m: "-".join(f"{k}{v}" for k, v in m.items()) or "plain")
def test_varlen_rising_scores(hq, hkv, bs, mod):
    q_lens, seq_lens = [700, 130, 1, 40], [700, 1000, 900, 600]
    case = rising_case(1200 + hq + bs, q_lens, seq_lens, hq, hkv, bs)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    sinks = torch.full((hq,), mod["sinks"], dtype=torch.float32) if "sinks" in mod else None
    kw = dict(window=mod.get("window", 0), softcap=mod.get("softcap", 0.0))
    want = oracle.paged_attention_varlen(case.q, ko, vo, case.query_start_loc, case.seq_lens, case.block_tables,
                                         True, case.scale, sinks=None if sinks is None else sinks.double(), **kw)
    for split in (False, True):
        out = pa.paged_attention_varlen(case.q.to(DEV), kc, vc, case.query_start_loc.to(DEV),
                                        case.seq_lens.to(DEV), case.block_tables.to(DEV), max(q_lens), True,
                                        case.scale, sinks=None if sinks is None else sinks.to(DEV),
                                        split_decodes=split, **kw)
        check_close(out, want, torch.bfloat16, label=f"rising varlen G{hq // hkv} bs{bs} {mod} split={split}")


@pytest.mark.gpu
@pytest.mark.parametrize("head_dim,hq,hkv,bs", [(64, 32, 8, 16), (64, 16, 1, 64), (256, 16, 4, 64),
                                                 (256, 8, 8, 16), (256, 16, 1, 32)])
@pytest.mark.parametrize("mod", MODS, ids=lambda m: "-".join(f"{k}{v}" for k, v in m.items()) or "plain")
def test_varlen_rising_scores_other_head_dims(head_dim, hq, hkv, bs, mod):
    """The same jumps on the head_dim 64 and 256 tensor-core kernels (at 256 a rescale of O waits
    for the previous tile's P.V, which may still be running when the next scores are ready)."""
    q_lens, seq_lens = [700, 130, 1, 40], [700, 1000, 900, 600]
    case = rising_case(1300 + head_dim + hq + bs, q_lens, seq_lens, hq, hkv, bs, head_dim)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    sinks = torch.full((hq,), mod["sinks"], dtype=torch.float32) if "sinks" in mod else None
    kw = dict(window=mod.get("window", 0), softcap=mod.get("softcap", 0.0))
    want = oracle.paged_attention_varlen(case.q, ko, vo, case.query_start_loc, case.seq_lens, case.block_tables,
                                         True, case.scale, sinks=None if sinks is None else sinks.double(), **kw)
    out = pa.paged_attention_varlen(case.q.to(DEV), kc, vc, case.query_start_loc.to(DEV), case.seq_lens.to(DEV),
                                    case.block_tables.to(DEV), max(q_lens), True, case.scale,
                                    sinks=None if sinks is None else sinks.to(DEV), **kw)
    check_close(out, want, torch.bfloat16, label=f"rising varlen D{head_dim} G{hq // hkv} bs{bs} {mod}")


@pytest.mark.gpu
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_decode_rising_scores(splits):
    case = rising_case(1250 + splits, [1] * 4, [1000, 700, 129, 1024], 32, 8, 16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    out = pa.paged_attention_decode(case.q.to(DEV), kc, vc, case.block_tables.to(DEV), case.seq_lens.to(DEV),
                                    case.scale, num_splits=splits)
    want = oracle.paged_attention_decode(case.q, ko, vo, case.block_tables, case.seq_lens, case.scale)
    check_close(out, want, torch.bfloat16, label=f"rising decode splits={splits}")


def test_rising_case_reaches_every_branch():
    """The data really holds the jumps the kernel's branches are for (checked on the CPU): some
    row's log2-unit maximum rises by 8-64 and by more than 64 from one key tile to a later one."""
    case = rising_case(1232, [700], [700], 32, 8, 16)
    G = 4
    # per head: log2-unit score maxima of key tiles 0..4 for the last query (it sees every key)
    qt = case.q.double()[-1]  # [Hq, D]
    kk = case.key.double().repeat_interleave(G, dim=1)  # [L, Hq, D]
    sc = torch.einsum("hd,lhd->hl", qt, kk) * case.scale * 1.4426950408889634
    m = [sc[:, 128 * i:128 * (i + 1)].max(dim=1).values for i in range(5)]
    rises = torch.stack([m[i + 1] - torch.stack(m[:i + 1]).max(0).values for i in range(4)])
    assert ((rises > 8) & (rises <= 64)).any()
    assert (rises > 64).any()
