"""GPU parity of pa_paged_attention_varlen (prefill chunks, decodes and verify blocks in one
flattened batch, causal by position) against the float64 oracle."""

import functools

import pytest
import torch

import oracle
import paged_kv_attention_gb300 as pa
import workloads
from paged_helpers import check_close, gpu_pools, named_case, oracle_pools

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_varlen(case, kc, vc, causal=None, **kw):
    return pa.paged_attention_varlen(case.q.to(DEV), kc, vc, case.query_start_loc.to(DEV),
                                     case.seq_lens.to(DEV), case.block_tables.to(DEV), case.max_query_len,
                                     case.causal if causal is None else causal, case.scale, **kw)


def oracle_varlen(case, ko, vo, causal=None, tokens=None):
    return oracle.paged_attention_varlen(case.q, ko, vo, case.query_start_loc, case.seq_lens,
                                         case.block_tables, case.causal if causal is None else causal,
                                         case.scale, tokens=tokens)


def sample_tokens(case, stride=23, edge=40):
    """Every decode / verify token, both ends of every long query block, and a stride sample."""
    qsl = case.query_start_loc.tolist()
    picked = set()
    for r in range(case.num_reqs):
        a, b = qsl[r], qsl[r + 1]
        if b - a <= 2 * edge:
            picked.update(range(a, b))
        else:
            picked.update(range(a, a + edge))
            picked.update(range(b - edge, b))
            picked.update(range(a, b, stride))
    return torch.tensor(sorted(picked))


@functools.lru_cache(maxsize=1)
def mixed_oracle_all_rows():
    case, (ko, vo) = named_case("varlen_mixed_bf16")
    return oracle_varlen(case, ko, vo)


@pytest.mark.parametrize("path", ["default", "split_decodes", "planned", "planned_split"])
def test_mixed_batch_every_row(path):
    """The mixed batch (8 prefill chunks of 512, 48 decodes, 8 verify blocks of 5: 4,184 rows x
    32 heads), every element against the oracle, on each of the call's grids."""
    case, _ = named_case("varlen_mixed_bf16")
    kc, vc = gpu_pools(case)
    split = path in ("split_decodes", "planned_split")
    kw = dict(split_decodes=split)
    if path.startswith("planned"):
        items = pa.varlen_plan(case.query_start_loc, case.seq_lens, case.max_query_len, case.num_q_heads,
                               case.num_kv_heads, case.causal, 0, split_decodes=split)
        kw["work_items"] = items.to(DEV)
    out = run_varlen(case, kc, vc, **kw)
    check_close(out, mixed_oracle_all_rows(), case.dtype, label=f"mixed ({path})")


def test_long_causal_prefill_one_whole_prompt():
    """The 4 x 8192 causal prefill: one whole prompt (all 8,192 rows x 32 heads) against the oracle;
    for the other three, every diagonal-tile row of their first and last tile pairs and a
    stride-17 sample; every row of all four finite."""
    case, (ko, vo) = named_case("prefill_4x8192_bf16")
    kc, vc = gpu_pools(case)
    out = run_varlen(case, kc, vc)
    qsl = case.query_start_loc.tolist()
    whole = torch.arange(qsl[1], qsl[2])                      # request 1, all rows
    check_close(out, oracle_varlen(case, ko, vo, tokens=whole), case.dtype, rows=whole,
                label="prefill 4x8192, request 1 whole")
    rows = sample_tokens(case, stride=17, edge=128)
    rows = rows[(rows < qsl[1]) | (rows >= qsl[2])]
    check_close(out, oracle_varlen(case, ko, vo, tokens=rows), case.dtype, rows=rows,
                label="prefill 4x8192, other requests sampled")
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("head_dim,hq,hkv,bs", [(128, 32, 8, 16), (128, 8, 8, 16), (64, 16, 2, 32),
                                                 (256, 8, 4, 64), (128, 16, 1, 64), (128, 4, 2, 128)])
@pytest.mark.parametrize("causal", [True, False])
def test_small_mixed_batches(dtype, head_dim, hq, hkv, bs, causal):
    if dtype == torch.float32 and (hq // hkv) * head_dim > 2048:
        pytest.skip("f32 path covers group * head_dim <= 2048")
    q_lens = [37, 1, 5, 0, 130, 16, 1]
    seq_lens = [90, 33, 64, 12, 130, 200, 1]
    case = workloads.make_case("vsmall", 300 + head_dim + hq + bs, q_lens, seq_lens, num_q_heads=hq,
                               num_kv_heads=hkv, head_dim=head_dim, block_size=bs, dtype=dtype, causal=causal)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    out = run_varlen(case, kc, vc)
    check_close(out, oracle_varlen(case, ko, vo), dtype, label=f"D{head_dim} G{hq // hkv} bs{bs} causal={causal}")


def test_qlen1_batch_matches_decode():
    case = workloads.decode_case("v1", 71, [5, 700, 33, 4000], num_q_heads=32, num_kv_heads=8, head_dim=128,
                                 block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    a = run_varlen(case, kc, vc)
    b = pa.paged_attention_decode(case.q.to(DEV), kc, vc, case.block_tables.to(DEV), case.seq_lens.to(DEV),
                                  case.scale, num_splits=1)
    diff = (a.float() - b.float()).abs().max().item()
    assert diff <= 2e-2


def test_chunked_prefill_matches_full_prefill():
    """The last chunk of a prompt, run as a chunk over its prior context, equals those rows
    of the full prompt's causal prefill."""
    L, chunk = 700, 180
    full = workloads.make_case("cf", 81, [L], [L], num_q_heads=32, num_kv_heads=8, head_dim=128,
                               block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(full)
    out_full = run_varlen(full, kc, vc)
    q_tail = full.q[L - chunk:].to(DEV)
    qsl = torch.tensor([0, chunk], dtype=torch.int32, device=DEV)
    out_chunk = pa.paged_attention_varlen(q_tail, kc, vc, qsl, full.seq_lens.to(DEV), full.block_tables.to(DEV),
                                          chunk, True, full.scale)
    diff = (out_chunk.float() - out_full[L - chunk:].float()).abs().max().item()
    assert diff <= 2e-2


def test_query_longer_than_context_is_flagged():
    case = workloads.make_case("bad", 91, [4, 3], [10, 20], num_q_heads=8, num_kv_heads=2, head_dim=128,
                               block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    bad_lens = case.seq_lens.clone()
    bad_lens[0] = 2                                   # q_len 4 > seq_len 2
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pa.paged_attention_varlen(case.q.to(DEV), kc, vc, case.query_start_loc.to(DEV), bad_lens.to(DEV),
                                    case.block_tables.to(DEV), case.max_query_len, True, case.scale,
                                    error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa._lib.PA_ERRBIT_QUERY_LAYOUT
    assert torch.equal(out[:4].float(), torch.zeros_like(out[:4].float()))
    ko, vo = oracle_pools(case)
    want = oracle_varlen(case, ko, vo)
    check_close(out[4:], want[4:], torch.bfloat16, label="clean request")


def test_cuda_graph_replay_follows_device_positions():
    """The varlen launch shape depends on host sizes only: a captured call replays correctly
    after seq_lens (a device buffer) grow, i.e. the queries move to later positions."""
    full = [700, 300, 1200]
    q_lens = [64, 1, 5]
    case = workloads.make_case("vg", 95, q_lens, full, num_q_heads=32, num_kv_heads=8, head_dim=128,
                               block_size=16, dtype=torch.bfloat16)
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
        want = oracle.paged_attention_varlen(case.q, ko, vo, case.query_start_loc, new, case.block_tables, True,
                                             case.scale)
        check_close(out, want, torch.bfloat16, label=f"varlen graph step {step}")


@pytest.mark.parametrize("split_decodes", [True, False])
@pytest.mark.parametrize("hq,hkv,bs", [(32, 8, 16), (16, 1, 64), (8, 8, 16)])
def test_one_query_requests_on_either_path(split_decodes, hq, hkv, bs):
    """One-query requests are served by the split-KV decode (with a workspace) or by the
    tensor-core kernel (without); both agree with the oracle, long contexts included."""
    q_lens = [1, 64, 1, 5, 1, 1, 200, 1]
    seq_lens = [3000, 100, 1, 900, 4096, 17, 700, 2500]
    case = workloads.make_case("v1q", 97 + hq + bs, q_lens, seq_lens, num_q_heads=hq, num_kv_heads=hkv,
                               head_dim=128, block_size=bs, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    out = run_varlen(case, kc, vc, split_decodes=split_decodes)
    rows = sample_tokens(case)
    check_close(out, oracle_varlen(case, ko, vo, tokens=rows), torch.bfloat16, rows=rows,
                label=f"split_decodes={split_decodes} G{hq // hkv} bs{bs}")


SHORT_Q = [2, 1, 5, 8, 9, 3, 64, 4, 7, 6]          # 9 and 64: past the short limit (8 queries)
SHORT_SEQ = [2, 3000, 900, 2500, 800, 40, 300, 4096, 17, 129]


@pytest.mark.parametrize("hq,hkv,bs", [(32, 8, 16), (16, 2, 64), (16, 1, 32), (8, 8, 16), (8, 4, 128)])
@pytest.mark.parametrize("causal", [True, False])
def test_short_requests_on_the_split_path(hq, hkv, bs, causal):
    """Requests of up to 8 queries (decodes, verify blocks) go to the split-KV decode in units of
    up to 16 query rows, each query seeing its own causal range; the rest of the batch stays on
    the tensor-core kernel. Every short request's every query is checked against the oracle."""
    case = workloads.make_case("vshort", 300 + hq + hkv + bs, SHORT_Q, SHORT_SEQ, num_q_heads=hq, num_kv_heads=hkv,
                               head_dim=128, block_size=bs, dtype=torch.bfloat16, causal=causal)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_varlen(case, kc, vc, split_decodes=True, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = sample_tokens(case)
    check_close(out, oracle_varlen(case, ko, vo, tokens=rows), torch.bfloat16, rows=rows,
                label=f"short requests G{hq // hkv} bs{bs} causal={causal}")
    # the same batch without the split path: the same rows within the tolerance of both paths
    ref = run_varlen(case, kc, vc, split_decodes=False)
    assert (out.float() - ref.float()).abs().max().item() <= 2e-2


@pytest.mark.parametrize("window,softcap,sinks", [(100, 0.0, False), (0, 30.0, False), (0, 0.0, True),
                                                  (37, 20.0, True)])
def test_short_requests_with_score_modifiers(window, softcap, sinks):
    case = workloads.make_case("vshortm", 411 + window, SHORT_Q, SHORT_SEQ, num_q_heads=32, num_kv_heads=8,
                               head_dim=128, block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    sk = torch.linspace(-2.0, 3.0, 32, dtype=torch.float32) if sinks else None
    out = run_varlen(case, kc, vc, split_decodes=True, window=window, softcap=softcap,
                     sinks=None if sk is None else sk.to(DEV))
    rows = sample_tokens(case)
    want = oracle.paged_attention_varlen(case.q, ko, vo, case.query_start_loc, case.seq_lens, case.block_tables,
                                         True, case.scale, tokens=rows, window=window, softcap=softcap, sinks=sk)
    check_close(out, want, torch.bfloat16, rows=rows, label=f"short w{window} cap{softcap} sinks{sinks}")


def test_short_request_without_its_positions_is_flagged_on_the_split_path():
    case = workloads.make_case("vse", 99, [3, 4], [10, 20], num_q_heads=8, num_kv_heads=2, head_dim=128,
                               block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    lens = case.seq_lens.clone()
    lens[0] = 2                                       # three queries but only two cached positions
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pa.paged_attention_varlen(case.q.to(DEV), kc, vc, case.query_start_loc.to(DEV), lens.to(DEV),
                                    case.block_tables.to(DEV), case.max_query_len, True, case.scale,
                                    error_word=err, split_decodes=True)
    torch.cuda.synchronize()
    assert int(err.item()) & pa._lib.PA_ERRBIT_QUERY_LAYOUT
    assert torch.equal(out[:3].float(), torch.zeros_like(out[:3].float()))
    ko, vo = oracle_pools(case)
    check_close(out[3:], oracle_varlen(case, ko, vo)[3:], torch.bfloat16, label="clean request")


@pytest.mark.parametrize("hq,hkv", [(32, 8), (12, 4), (8, 8)])   # group 4, group 3, MHA
@pytest.mark.parametrize("window", [0, 24])
def test_milestone_batch_matches_each_request_alone(hq, hkv, window):
    """The milestone batch of 32. Production attention kernels, "The tests and the measurements": a prefill
    chunk in the middle of its prompt, a whole 16-token prompt, a 21-token prompt and decodes at
    70 and 130 cached tokens, in one batch. Every row matches the oracle, and every request's rows
    equal (bit for bit) what the same call gives for that request alone."""
    q_lens = [32, 16, 21, 1, 1]
    seq_lens = [72, 16, 21, 70, 130]
    case = workloads.make_case("milestone", 500 + hq + window, q_lens, seq_lens, num_q_heads=hq, num_kv_heads=hkv,
                               head_dim=128, block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    out = run_varlen(case, kc, vc, window=window)
    want = oracle.paged_attention_varlen(case.q, ko, vo, case.query_start_loc, case.seq_lens, case.block_tables,
                                         True, case.scale, window=window)
    check_close(out, want, torch.bfloat16, label=f"milestone Hq{hq} Hkv{hkv} w{window}")
    qsl = case.query_start_loc.tolist()
    for r in range(len(q_lens)):
        a, b = qsl[r], qsl[r + 1]
        solo = pa.paged_attention_varlen(case.q[a:b].to(DEV), kc, vc,
                                         torch.tensor([0, b - a], dtype=torch.int32, device=DEV),
                                         case.seq_lens[r:r + 1].to(DEV), case.block_tables[r:r + 1].to(DEV),
                                         case.max_query_len, True, case.scale, window=window)
        assert torch.equal(solo, out[a:b]), f"request {r} differs alone"


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("window", [0, 700])
def test_planned_grid_equals_default_grid(split, window):
    """pa_varlen_plan + pa_paged_attention_varlen_planned: only the pairs the batch has, longest
    first. Each pair's CTA computes what it computes on the default grid: bitwise equal."""
    case, _ = named_case("varlen_mixed_bf16")
    kc, vc = gpu_pools(case)
    items = pa.varlen_plan(case.query_start_loc, case.seq_lens, case.max_query_len, case.num_q_heads,
                           case.num_kv_heads, case.causal, window, split_decodes=split)
    assert 0 < items.numel() < case.num_reqs * -(-case.max_query_len // 64)
    base = run_varlen(case, kc, vc, split_decodes=split, window=window)
    planned = run_varlen(case, kc, vc, split_decodes=split, window=window, work_items=items.to(DEV))
    assert torch.equal(base, planned)


@pytest.mark.parametrize("hq,hkv,bs", [(32, 8, 16), (16, 1, 64), (8, 8, 128), (16, 2, 32)])
def test_planned_small_batches(hq, hkv, bs):
    q_lens, seq_lens = [1, 64, 0, 37, 130, 5, 300], [700, 100, 3, 37, 900, 5, 2000]
    case = workloads.make_case("vplan", 700 + hq + bs, q_lens, seq_lens, num_q_heads=hq, num_kv_heads=hkv,
                               head_dim=128, block_size=bs, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    items = pa.varlen_plan(case.query_start_loc, case.seq_lens, case.max_query_len, hq, hkv)
    out = run_varlen(case, kc, vc, work_items=items.to(DEV))
    assert torch.equal(out, run_varlen(case, kc, vc))
    rows = sample_tokens(case)
    check_close(out, oracle_varlen(case, ko, vo, tokens=rows), torch.bfloat16, rows=rows, label="planned")


def test_plan_item_outside_the_batch_is_flagged():
    case = workloads.make_case("vplanbad", 77, [40, 3], [40, 10], num_q_heads=8, num_kv_heads=2, head_dim=128,
                               block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    items = pa.varlen_plan(case.query_start_loc, case.seq_lens, case.max_query_len, 8, 2)
    bad = torch.cat([items, torch.tensor([99 * case.num_reqs], dtype=torch.int32)]).to(DEV)  # tile 99
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_varlen(case, kc, vc, work_items=bad, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa._lib.PA_ERRBIT_QUERY_LAYOUT
    assert torch.equal(out, run_varlen(case, kc, vc))


def test_one_query_request_without_its_position_is_flagged():
    case = workloads.make_case("v1e", 98, [1, 3], [10, 20], num_q_heads=8, num_kv_heads=2, head_dim=128,
                               block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    lens = case.seq_lens.clone()
    lens[0] = 0                                       # the query's own position is not cached
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pa.paged_attention_varlen(case.q.to(DEV), kc, vc, case.query_start_loc.to(DEV), lens.to(DEV),
                                    case.block_tables.to(DEV), case.max_query_len, True, case.scale,
                                    error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa._lib.PA_ERRBIT_QUERY_LAYOUT
    assert torch.equal(out[:1].float(), torch.zeros_like(out[:1].float()))
    ko, vo = oracle_pools(case)
    check_close(out[1:], oracle_varlen(case, ko, vo)[1:], torch.bfloat16, label="clean request")


@pytest.mark.parametrize("hq,hkv,bs", [(32, 8, 16), (16, 4, 64), (16, 1, 32)])
def test_device_planned_grid_follows_the_batch_under_graph_replay(hq, hkv, bs):
    """With a workspace the tensor-core grid is planned on the device from the lengths as they
    are when the call runs: a captured call replays correctly after both seq_lens and the query
    layout (query_start_loc, same total) change, prefill chunks turning into decodes and back."""
    layouts = [([300, 1, 5, 60, 1, 200], [900, 3000, 1100, 60, 17, 2500]),
               ([1, 1, 500, 5, 60, 0], [40, 2600, 1500, 1200, 300, 10]),
               ([8, 9, 1, 230, 318, 1], [8, 700, 2999, 230, 1400, 64])]
    N = sum(layouts[0][0])
    assert all(sum(q) == N for q, _ in layouts)
    max_q = 512
    width = 3000 // bs + 1
    pool = max(sum(-(-x // bs) for x in L) for _, L in layouts) + 8   # one pool size for every layout
    cases = [workloads.make_case("vdp", 3100 + i + hq + bs, q, L, num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                                 block_size=bs, dtype=torch.bfloat16, pool_blocks=pool, table_multiple=width)
             for i, (q, L) in enumerate(layouts)]
    # one pool per layout, one set of device buffers the graph reads
    q = torch.empty((N, hq, 128), dtype=torch.bfloat16, device=DEV)
    qsl = torch.empty(len(layouts[0][0]) + 1, dtype=torch.int32, device=DEV)
    lens = torch.empty(len(layouts[0][0]), dtype=torch.int32, device=DEV)
    tables = torch.empty((len(layouts[0][0]), cases[0].block_tables.shape[1]), dtype=torch.int32, device=DEV)
    pools = [gpu_pools(c) for c in cases]
    kc = torch.empty_like(pools[0][0])
    vc = torch.empty_like(pools[0][1])
    out = torch.empty_like(q)
    ws = torch.empty(max(pa._lib.load().pa_varlen_workspace_bytes(len(lens), hq, 128, tables.shape[1], bs), 16),
                     dtype=torch.uint8, device=DEV)

    def load(i):
        c = cases[i]
        q.copy_(c.q.to(DEV))
        qsl.copy_(c.query_start_loc.to(DEV))
        lens.copy_(c.seq_lens.to(DEV))
        tables.copy_(c.block_tables.to(DEV))
        kc.copy_(pools[i][0])
        vc.copy_(pools[i][1])

    def call():
        pa.paged_attention_varlen(q, kc, vc, qsl, lens, tables, max_q, True, cases[0].scale, out=out, workspace=ws,
                                  split_decodes=True)

    load(0)
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for i in (1, 2, 0):
        load(i)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ko, vo = oracle_pools(cases[i])
        check_close(out, oracle_varlen(cases[i], ko, vo), torch.bfloat16, label=f"device plan replay layout {i}")


@pytest.mark.parametrize("hq,hkv,bs", [(32, 8, 16), (16, 2, 64)])
def test_schedules(hq, hkv, bs):
    """pa_paged_attention_varlen_sched: "tensor" (device-planned grid, every request on the tensor
    cores) equals the default grid bit for bit; "split" equals the split path; "auto" picks the
    split-KV decode for a batch of many short requests (>= 80 requests, <= 8 queries each on
    average) and the tensor-core kernel otherwise; all agree with the oracle."""
    heavy = workloads.make_case("vsch", 3200 + hq + bs, [300, 1, 5, 130, 1, 64], [900, 3000, 1100, 130, 17, 2500],
                                num_q_heads=hq, num_kv_heads=hkv, head_dim=128, block_size=bs, dtype=torch.bfloat16)
    gen = torch.Generator().manual_seed(3300 + hq + bs)
    lq = [1, 5, 2, 1, 8, 3] * 14 + [20]
    ls = [int(x) for x in torch.randint(120, 1500, (len(lq),), generator=gen)]
    light = workloads.make_case("vsch", 3300 + hq + bs, lq, ls, num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                                block_size=bs, dtype=torch.bfloat16)
    assert heavy.num_reqs < 80 and light.num_reqs >= 80 and light.num_tokens <= 8 * light.num_reqs
    for case in (heavy, light):
        kc, vc = gpu_pools(case)
        ko, vo = oracle_pools(case)
        grid = run_varlen(case, kc, vc)
        tensor = run_varlen(case, kc, vc, schedule="tensor")
        split = run_varlen(case, kc, vc, schedule="split")
        auto = run_varlen(case, kc, vc, schedule="auto")
        assert torch.equal(grid, tensor)
        assert torch.equal(auto, split if case is light else tensor)
        want = oracle_varlen(case, ko, vo)
        check_close(tensor, want, torch.bfloat16, label="tensor schedule")
        check_close(split, want, torch.bfloat16, label="split schedule")


def test_split_schedule_without_workspace_is_refused():
    case = workloads.make_case("vschw", 3400, [3, 1], [10, 20], num_q_heads=8, num_kv_heads=2, head_dim=128,
                               block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    lib = pa._lib.load()
    out = torch.empty_like(case.q.to(DEV))
    st = lib.pa_paged_attention_varlen_sched(
        case.q.to(DEV).data_ptr(), kc.data_ptr(), vc.data_ptr(), case.query_start_loc.to(DEV).data_ptr(),
        case.seq_lens.to(DEV).data_ptr(), case.block_tables.to(DEV).data_ptr(), 2, 4, 3, 8, 2, 128, 16,
        case.num_blocks, case.block_tables.shape[1], 1, 0.0, pa._lib.PA_DTYPE_BF16, out.data_ptr(), None, None,
        pa._lib.PA_SHORT_SPLIT, None, 0, None, None)
    assert st == pa._lib.PA_ERR_WORKSPACE_TOO_SMALL


# Lone query tiles: a pair whose second tile is empty splits its key tiles between the two softmax
# groups (even tiles one group, odd tiles the other) over a three-stage K/V ring, and merges the two
# partial states at the end. Key-tile counts 1 to 9 and 33 cover the single-group case, the ring's
# wrap at every phase, and the merge; 2 * TOK + 5 queries give a full pair followed by a lone one.
@pytest.mark.parametrize("head_dim,hq,hkv,bs", [(128, 32, 8, 16), (128, 16, 1, 128), (64, 16, 2, 32),
                                                (128, 64, 4, 64)])
@pytest.mark.parametrize("window,softcap,sinks", [(0, 0.0, False), (150, 25.0, True)])
def test_lone_tiles(head_dim, hq, hkv, bs, window, softcap, sinks):
    tok = 128 // (hq // hkv)
    keys = [1, 128, 129, 256, 300, 384, 513, 640, 900, 1152, 4200]
    q_lens = [1, tok, 5, 1, tok - 1, 3, 1, tok, 2, 7, 1] + [2 * tok + 5]
    seq_lens = keys + [1500]
    case = workloads.make_case("vlone", 7100 + head_dim + hq + bs, q_lens, seq_lens, num_q_heads=hq,
                               num_kv_heads=hkv, head_dim=head_dim, block_size=bs, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    sk = torch.linspace(-1.0, 2.5, hq, dtype=torch.float32) if sinks else None
    out = run_varlen(case, kc, vc, window=window, softcap=softcap, sinks=None if sk is None else sk.to(DEV))
    want = oracle.paged_attention_varlen(case.q, ko, vo, case.query_start_loc, case.seq_lens, case.block_tables,
                                         True, case.scale, window=window, softcap=softcap, sinks=sk)
    check_close(out, want, torch.bfloat16, label=f"lone D{head_dim} G{hq // hkv} bs{bs} w{window}")
