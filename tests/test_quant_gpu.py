"""GPU parity of the 8-bit KV cache: the quantising write is bit-exact against the oracle's
quantiser (same float32 arithmetic), and decode / varlen over int8 and fp8 pools match the
float64 attention over the oracle's dequantised cache within the bf16 tolerance."""

import pytest
import torch

import paged_kv_attention_gb300 as pa
import workloads
from oracle import quant
from paged_helpers import check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
KINDS = {"int8": torch.int8, "fp8": torch.float8_e4m3fn}


def pools(case, kind, dev):
    shape = (case.num_blocks, case.block_size, case.num_kv_heads, case.head_dim)
    kc = torch.zeros(shape, dtype=KINDS[kind], device=dev)
    vc = torch.zeros(shape, dtype=KINDS[kind], device=dev)
    # scales of unwritten slots are NaN: a kernel that reads one shows it
    ks = torch.full(shape[:3], float("nan"), dtype=torch.float32, device=dev)
    vs = torch.full(shape[:3], float("nan"), dtype=torch.float32, device=dev)
    return kc, vc, ks, vs


def filled(case, kind):
    g = pools(case, kind, DEV)
    pa.reshape_and_cache_quant(case.key.to(DEV), case.value.to(DEV), *g, case.slot_mapping.to(DEV))
    o = pools(case, kind, "cpu")
    quant.reshape_and_cache_quant(case.key, case.value, *o, case.slot_mapping, kind)
    return g, o


def _bits(t):
    return t.view(torch.uint8) if t.element_size() == 1 else t.view(torch.int32)


@pytest.mark.parametrize("kind", ["int8", "fp8"])
@pytest.mark.parametrize("src", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("hkv,d", [(8, 128), (4, 256), (2, 64)])
def test_quantizing_write_is_bit_exact(kind, src, hkv, d):
    case = workloads.make_case("qw", 700 + d, [1, 1, 1], [37, 300, 5], num_q_heads=hkv, num_kv_heads=hkv,
                               head_dim=d, block_size=16, dtype=src)
    slots = case.slot_mapping.clone()
    slots[::9] = -1
    case.slot_mapping = slots
    g, o = filled(case, kind)
    torch.cuda.synchronize()
    for a, b in zip(g, o):
        assert torch.equal(_bits(a.cpu()), _bits(b))


@pytest.mark.parametrize("kind", ["int8", "fp8"])
@pytest.mark.parametrize("head_dim,hq,hkv", [(128, 32, 8), (256, 16, 4), (128, 16, 1), (128, 8, 8)])
@pytest.mark.parametrize("splits", [1, 4, 0])
def test_decode(kind, head_dim, hq, hkv, splits):
    case = workloads.decode_case("qd", 710 + head_dim + hq, [1, 15, 16, 17, 300, 2049], num_q_heads=hq,
                                 num_kv_heads=hkv, head_dim=head_dim, block_size=16, dtype=torch.bfloat16)
    (kc, vc, ks, vs), (ko, vo, kso, vso) = filled(case, kind)
    out = pa.paged_attention_decode_quant(case.q.to(DEV), kc, vc, ks, vs, case.block_tables.to(DEV),
                                          case.seq_lens.to(DEV), case.scale, num_splits=splits)
    want = quant.paged_attention_decode_quant(case.q, ko, vo, kso, vso, case.block_tables, case.seq_lens, case.scale)
    check_close(out, want, torch.bfloat16, label=f"{kind} D{head_dim} G{hq // hkv} splits={splits}")


@pytest.mark.parametrize("kind", ["int8", "fp8"])
def test_decode_with_modifiers(kind):
    case = workloads.decode_case("qm", 720, [40, 333, 1500], num_q_heads=16, num_kv_heads=4, head_dim=128,
                                 block_size=32, dtype=torch.bfloat16)
    (kc, vc, ks, vs), (ko, vo, kso, vso) = filled(case, kind)
    sinks = torch.randn(16, generator=torch.Generator().manual_seed(1))
    out = pa.paged_attention_decode_quant(case.q.to(DEV), kc, vc, ks, vs, case.block_tables.to(DEV),
                                          case.seq_lens.to(DEV), case.scale, window=100, softcap=4.0,
                                          sinks=sinks.to(DEV))
    want = quant.paged_attention_decode_quant(case.q, ko, vo, kso, vso, case.block_tables, case.seq_lens, case.scale,
                                              window=100, softcap=4.0, sinks=sinks.double())
    check_close(out, want, torch.bfloat16, label=f"{kind} modifiers")


@pytest.mark.parametrize("kind", ["int8", "fp8"])
def test_varlen(kind):
    case = workloads.make_case("qv", 730, [37, 1, 5, 0, 64], [90, 33, 64, 12, 64], num_q_heads=32, num_kv_heads=8,
                               head_dim=128, block_size=16, dtype=torch.bfloat16)
    (kc, vc, ks, vs), (ko, vo, kso, vso) = filled(case, kind)
    out = pa.paged_attention_varlen_quant(case.q.to(DEV), kc, vc, ks, vs, case.query_start_loc.to(DEV),
                                          case.seq_lens.to(DEV), case.block_tables.to(DEV), case.max_query_len,
                                          True, case.scale)
    want = quant.paged_attention_varlen_quant(case.q, ko, vo, kso, vso, case.query_start_loc, case.seq_lens,
                                              case.block_tables, True, case.scale)
    check_close(out, want, torch.bfloat16, label=f"{kind} varlen")


def test_64x4096_int8_decode_full_size():
    case = workloads.NAMED["decode_64x4096_bf16"]()
    (kc, vc, ks, vs), (ko, vo, kso, vso) = filled(case, "int8")
    out = pa.paged_attention_decode_quant(case.q.to(DEV), kc, vc, ks, vs, case.block_tables.to(DEV),
                                          case.seq_lens.to(DEV), case.scale)
    want = quant.paged_attention_decode_quant(case.q, ko, vo, kso, vso, case.block_tables, case.seq_lens, case.scale)
    check_close(out, want, torch.bfloat16, label="int8 64x4096")


def test_unsupported_head_dim_is_refused():
    case = workloads.decode_case("qx", 740, [10], num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
                                 dtype=torch.bfloat16)
    (kc, vc, ks, vs), _ = filled(case, "int8")
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.paged_attention_decode_quant(case.q.to(DEV), kc, vc, ks, vs, case.block_tables.to(DEV),
                                        case.seq_lens.to(DEV), case.scale)
    assert e.value.status == pa._lib.PA_ERR_UNSUPPORTED


@pytest.mark.parametrize("kind", ["int8", "fp8"])
@pytest.mark.parametrize("keys", ["alike", "random"])
def test_decode_long_diffuse_attention_with_one_sign_queries(kind, keys):
    """Cases where a shortcut in the 8-bit arithmetic would show. The int8 codes enter the MMAs
    offset by 1152 and the offsets come out of the sums afterwards: out of each score, 1152 times
    the query row's dim sum, largest against the scores when every query dim has one sign and the
    keys are random ("random"); out of P.V, 1152 times the probability sum, largest against the
    output when the keys are alike, so that every probability is near 1 over 8,192 keys and the
    output is a weighted mean of values close to 0 ("alike"). Against the float64 attention over
    the dequantised cache (E4M3 alike, as a control)."""
    case = workloads.decode_case("qo", 750, [8192, 4096, 17, 1], num_q_heads=32, num_kv_heads=8, head_dim=128,
                                 block_size=16, dtype=torch.bfloat16)
    g = torch.Generator().manual_seed(751)
    case.q = (case.q.float().abs() + 1.0).to(torch.bfloat16)
    if keys == "alike":
        case.key = (1.0 + 0.01 * torch.randn(case.key.shape, generator=g)).to(torch.bfloat16)
    (kc, vc, ks, vs), (ko, vo, kso, vso) = filled(case, kind)
    out = pa.paged_attention_decode_quant(case.q.to(DEV), kc, vc, ks, vs, case.block_tables.to(DEV),
                                          case.seq_lens.to(DEV), case.scale, num_splits=1)
    want = quant.paged_attention_decode_quant(case.q, ko, vo, kso, vso, case.block_tables, case.seq_lens, case.scale)
    mx, _ = check_close(out, want, torch.bfloat16, label=f"{kind} {keys} keys, one-sign queries")
    if keys == "alike":
        # the 8,192-key row: a mean of ~8,192 values, so close to 0; its error stays far below
        # the bf16 budget (the offset's rounding, ~1152 x the values' scale x 2^-24 per add)
        err = (out[0].double().cpu() - want[0]).abs().max().item()
        assert err <= 2e-3, f"{kind} alike keys, 8192-key row: max abs {err:.3e}"


Q_LENS = [37, 1, 5, 0, 130, 300, 64, 1, 129]
SEQ_LENS = [90, 700, 2000, 3, 900, 300, 1000, 17, 129]


@pytest.mark.parametrize("kind", ["int8", "fp8"])
@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("bs", [16, 32, 64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_varlen_tensor_core_shapes(kind, G, bs, causal):
    """8-bit caches on the tensor-core varlen kernel (head_dim 128): each K / V tile's codes are
    dequantised in shared memory and used like a bf16 tile; every row against the oracle over the
    dequantised cache, for every group and block size, causal and not."""
    hkv = 2 if G <= 8 else 1
    case = workloads.make_case("qvt", 760 + 10 * G + bs, Q_LENS, SEQ_LENS, num_q_heads=G * hkv, num_kv_heads=hkv,
                               head_dim=128, block_size=bs, dtype=torch.bfloat16)
    (kc, vc, ks, vs), (ko, vo, kso, vso) = filled(case, kind)
    out = pa.paged_attention_varlen_quant(case.q.to(DEV), kc, vc, ks, vs, case.query_start_loc.to(DEV),
                                          case.seq_lens.to(DEV), case.block_tables.to(DEV), case.max_query_len,
                                          causal, case.scale)
    want = quant.paged_attention_varlen_quant(case.q, ko, vo, kso, vso, case.query_start_loc, case.seq_lens,
                                              case.block_tables, causal, case.scale)
    check_close(out, want, torch.bfloat16, label=f"{kind} varlen G{G} bs{bs} causal={causal}")


@pytest.mark.parametrize("kind", ["int8", "fp8"])
@pytest.mark.parametrize("window,softcap,sinks", [(100, 0.0, False), (0, 30.0, False), (0, 0.0, True),
                                                  (37, 20.0, True)])
def test_varlen_tensor_core_modifiers(kind, window, softcap, sinks):
    case = workloads.make_case("qvm", 800 + window, Q_LENS, SEQ_LENS, num_q_heads=32, num_kv_heads=8, head_dim=128,
                               block_size=16, dtype=torch.bfloat16)
    (kc, vc, ks, vs), (ko, vo, kso, vso) = filled(case, kind)
    sk = torch.linspace(-2.0, 3.0, 32, dtype=torch.float32) if sinks else None
    out = pa.paged_attention_varlen_quant(case.q.to(DEV), kc, vc, ks, vs, case.query_start_loc.to(DEV),
                                          case.seq_lens.to(DEV), case.block_tables.to(DEV), case.max_query_len,
                                          True, case.scale, window=window, softcap=softcap,
                                          sinks=None if sk is None else sk.to(DEV))
    want = quant.paged_attention_varlen_quant(case.q, ko, vo, kso, vso, case.query_start_loc, case.seq_lens,
                                              case.block_tables, True, case.scale, window=window, softcap=softcap,
                                              sinks=sk)
    check_close(out, want, torch.bfloat16, label=f"{kind} varlen w{window} cap{softcap} sinks{sinks}")


@pytest.mark.parametrize("kind", ["int8", "fp8"])
def test_varlen_long_prompt_and_head_dim_256(kind):
    """A 3,000-token causal prompt plus a 1,000-token chunk on the tensor-core path (every row), and
    the head_dim-256 shape, which runs as per-token decodes over the codes."""
    case = workloads.make_case("qvl", 830, [3000, 1000], [3000, 3000], num_q_heads=32, num_kv_heads=8, head_dim=128,
                               block_size=64, dtype=torch.bfloat16)
    (kc, vc, ks, vs), (ko, vo, kso, vso) = filled(case, kind)
    out = pa.paged_attention_varlen_quant(case.q.to(DEV), kc, vc, ks, vs, case.query_start_loc.to(DEV),
                                          case.seq_lens.to(DEV), case.block_tables.to(DEV), case.max_query_len,
                                          True, case.scale)
    want = quant.paged_attention_varlen_quant(case.q, ko, vo, kso, vso, case.query_start_loc, case.seq_lens,
                                              case.block_tables, True, case.scale)
    check_close(out, want, torch.bfloat16, label=f"{kind} varlen long")
    c2 = workloads.make_case("qv256", 831, [37, 1, 130], [90, 700, 400], num_q_heads=16, num_kv_heads=4,
                             head_dim=256, block_size=16, dtype=torch.bfloat16)
    (kc, vc, ks, vs), (ko, vo, kso, vso) = filled(c2, kind)
    out = pa.paged_attention_varlen_quant(c2.q.to(DEV), kc, vc, ks, vs, c2.query_start_loc.to(DEV),
                                          c2.seq_lens.to(DEV), c2.block_tables.to(DEV), c2.max_query_len, True,
                                          c2.scale)
    want = quant.paged_attention_varlen_quant(c2.q, ko, vo, kso, vso, c2.query_start_loc, c2.seq_lens,
                                              c2.block_tables, True, c2.scale)
    check_close(out, want, torch.bfloat16, label=f"{kind} varlen D256")


# Automatic splitting of an 8-bit decode at head_dim 128 (groups <= 8) runs as balanced segments:
# every resident CTA of a KV head streams the same share of the batch's chunks, sequences cut between
# CTAs are merged by the combine. These cases put sequence boundaries everywhere relative to the CTA
# ranges: empty contexts, one-chunk contexts, one long sequence spread over every CTA, thousands of
# short ones.
SEG_LENS = {
    "ragged": [1, 15, 16, 17, 300, 2049, 0, 4096, 33, 0, 1000, 7],
    "one_long": [8191],
    "many_short": [int(x) for x in torch.randint(0, 70, (3000,), generator=torch.Generator().manual_seed(5))],
    "uniform": [4096] * 24,
}


@pytest.mark.parametrize("kind", ["int8", "fp8"])
@pytest.mark.parametrize("lens", list(SEG_LENS))
@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (16, 2)])
def test_decode_balanced_segments(kind, lens, hq, hkv):
    L = SEG_LENS[lens]
    case = workloads.decode_case("qseg", 900 + len(L) + hq, L, num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                                 block_size=16, dtype=torch.bfloat16)
    (kc, vc, ks, vs), (ko, vo, kso, vso) = filled(case, kind)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pa.paged_attention_decode_quant(case.q.to(DEV), kc, vc, ks, vs, case.block_tables.to(DEV),
                                          case.seq_lens.to(DEV), case.scale, num_splits=0, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    seqs = list(range(case.num_reqs)) if case.num_reqs <= 64 else list(range(0, case.num_reqs, 7))
    want = quant.paged_attention_decode_quant(case.q, ko, vo, kso, vso, case.block_tables, case.seq_lens, case.scale,
                                              seqs=seqs)
    rows = torch.tensor(seqs)
    check_close(out, want, torch.bfloat16, rows=rows, label=f"{kind} segments {lens} G{hq // hkv}")
    empty = [s for s in seqs if L[s] == 0]
    if empty:
        assert torch.equal(out[empty].float(), torch.zeros_like(out[empty].float()))
    # the explicit one-split grid computes the same rows within the tolerance
    ref = pa.paged_attention_decode_quant(case.q.to(DEV), kc, vc, ks, vs, case.block_tables.to(DEV),
                                          case.seq_lens.to(DEV), case.scale, num_splits=1)
    assert (out.float() - ref.float()).abs().max().item() <= 2e-2


@pytest.mark.parametrize("kind", ["int8", "fp8"])
def test_decode_balanced_segments_with_modifiers_and_graph_replay(kind):
    """Window, softcap and sinks on the segment path; a captured call replays correctly after the
    context lengths change (the segments are recomputed from the device lengths at every run)."""
    full = [3000, 40, 1500, 0, 2222, 17]
    case = workloads.decode_case("qsegm", 930, full, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=32,
                                 dtype=torch.bfloat16)
    (kc, vc, ks, vs), (ko, vo, kso, vso) = filled(case, kind)
    sinks = torch.randn(32, generator=torch.Generator().manual_seed(2))
    sinks_dev = sinks.to(DEV)  # (a host-to-device copy inside the capture would invalidate it)
    q, tables = case.q.to(DEV), case.block_tables.to(DEV)
    lens = torch.tensor([1000, 40, 1500, 0, 2000, 1], dtype=torch.int32, device=DEV)
    out = torch.empty_like(q)
    ws = torch.empty(pa.decode_workspace_bytes(6, 32, 128, tables.shape[1], 32, 0), dtype=torch.uint8, device=DEV)

    def call():
        pa.paged_attention_decode_quant(q, kc, vc, ks, vs, tables, lens, case.scale, out=out, workspace=ws,
                                        window=700, softcap=30.0, sinks=sinks_dev)
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for new in ([1000, 40, 1500, 0, 2000, 1], [3000, 1, 900, 5, 2222, 17], [0, 0, 0, 0, 0, 8]):
        lens.copy_(torch.tensor(new, dtype=torch.int32))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        want = quant.paged_attention_decode_quant(case.q, ko, vo, kso, vso, case.block_tables,
                                                  torch.tensor(new, dtype=torch.int32), case.scale, window=700,
                                                  softcap=30.0, sinks=sinks.double())
        check_close(out, want, torch.bfloat16, label=f"{kind} segments replay {new}")
