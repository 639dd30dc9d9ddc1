"""The allocation-free decode entry point (pa_paged_attention_decode_static_scratch).

It is meant for callers that cannot allocate device memory (a plugin given only its input
and output pointers, a runtime that forbids cudaMalloc after start-up, a loop that cannot
pay cudaMalloc's device synchronisation); its split partials live in a fixed array inside
the library. Here it is called through the C ABI and checked against the regular entry
point on two calls in a row (the second call must not see the first one's leftovers), and
its size limit is checked. This file is collected last on purpose.
"""

import ctypes

import pytest
import torch

import paged_kv_attention_gb300 as pa
import workloads
from paged_helpers import TOL, gpu_pools
from paged_kv_attention_gb300 import _lib

pytestmark = pytest.mark.gpu
DEV = "cuda"
STATIC_SCRATCH_BYTES = 16 << 20


def _static_call(lib, q, kc, vc, tables, lens, out, scale, num_splits, dtype_code):
    S, Hq, D = q.shape
    nb, bs, Hkv = kc.shape[0], kc.shape[1], kc.shape[2]
    return lib.pa_paged_attention_decode_static_scratch(
        q.data_ptr(), kc.data_ptr(), vc.data_ptr(), tables.data_ptr(), lens.data_ptr(), S, Hq, Hkv, D, bs, nb,
        tables.shape[1], ctypes.c_float(scale), dtype_code, num_splits, out.data_ptr(), None,
        torch.cuda.current_stream().cuda_stream)


def _assert_within_tolerance(got, want, dtype):
    diff = (got.double() - want.double()).abs()
    assert torch.isfinite(got.float()).all()
    assert diff.max().item() <= TOL[dtype]["max_abs"]
    assert diff.mean().item() <= TOL[dtype]["mean_abs"]


def test_matches_the_regular_entry_on_two_calls_in_a_row():
    lib = _lib.load()
    case = workloads.decode_case("noalloc", 501, [2000, 700, 4096, 1, 333, 3000], num_q_heads=32,
                                 num_kv_heads=8, head_dim=128, block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    q = case.q.to(DEV)
    tables = case.block_tables.to(DEV)
    # call 1: full lengths, 8 splits; call 2: other lengths and queries, automatic split count,
    # so the scratch still holds call 1's partials when call 2 starts
    plans = [(case.seq_lens.to(DEV), q, 8),
             (torch.tensor([17, 650, 1, 1, 64, 1024], dtype=torch.int32, device=DEV), q.flip(0).contiguous(), 0)]
    for lens, qq, splits in plans:
        out = torch.empty_like(qq)
        st = _static_call(lib, qq, kc, vc, tables, lens, out, case.scale, splits, _lib.PA_DTYPE_BF16)
        assert st == _lib.PA_OK, pa.status_string(st)
        ref = pa.paged_attention_decode(qq, kc, vc, tables, lens, case.scale, num_splits=splits)
        torch.cuda.synchronize()
        _assert_within_tolerance(out, ref, torch.bfloat16)


def test_fp32_matches_the_regular_entry():
    lib = _lib.load()
    case = workloads.decode_case("noalloc32", 502, [200, 901, 50], num_q_heads=8, num_kv_heads=2, head_dim=64,
                                 block_size=16, dtype=torch.float32)
    kc, vc = gpu_pools(case)
    q, tables, lens = case.q.to(DEV), case.block_tables.to(DEV), case.seq_lens.to(DEV)
    for _ in range(2):
        out = torch.empty_like(q)
        assert _static_call(lib, q, kc, vc, tables, lens, out, case.scale, 4, _lib.PA_DTYPE_F32) == _lib.PA_OK
        ref = pa.paged_attention_decode(q, kc, vc, tables, lens, case.scale, num_splits=4)
        torch.cuda.synchronize()
        _assert_within_tolerance(out, ref, torch.float32)


def test_batches_beyond_the_fixed_scratch_are_refused():
    lib = _lib.load()
    S, Hq, Hkv, D, bs, mb = 64, 32, 8, 128, 16, 256
    need = pa.decode_workspace_bytes(S, Hq, D, mb, bs, 32)
    assert need > STATIC_SCRATCH_BYTES
    q = torch.zeros((S, Hq, D), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((4, bs, Hkv, D), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    tables = torch.zeros((S, mb), dtype=torch.int32, device=DEV)
    lens = torch.ones(S, dtype=torch.int32, device=DEV)
    out = torch.empty_like(q)
    st = _static_call(lib, q, kc, vc, tables, lens, out, 0.0, 32, _lib.PA_DTYPE_BF16)
    assert st == _lib.PA_ERR_WORKSPACE_TOO_SMALL
    # one split needs no scratch: the same batch is served
    assert _static_call(lib, q, kc, vc, tables, lens, out, 0.0, 1, _lib.PA_DTYPE_BF16) == _lib.PA_OK
    torch.cuda.synchronize()
