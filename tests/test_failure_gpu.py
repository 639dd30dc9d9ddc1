"""Failure detection on the GPU without a fault: a bounded wait that nothing completes expires,
reports PA_ERRBIT_WAIT_TIMEOUT through the error word, and the context stays usable."""

import time

import pytest
import torch

import paged_kv_attention_gb300 as pa
import workloads
from paged_helpers import check_close, gpu_pools, oracle_pools
from paged_kv_attention_gb300 import _lib
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_expired_wait_is_reported_and_the_context_survives():
    lib = _lib.load()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    t0 = time.perf_counter()
    st = lib.pa_selftest_wait_timeout(20000, err.data_ptr(), torch.cuda.current_stream().cuda_stream)  # 20 ms
    assert st == _lib.PA_OK
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(err.item()) == _lib.PA_ERRBIT_WAIT_TIMEOUT
    assert 0.015 < waited < 5.0
    # the context still runs real work afterwards
    case = workloads.decode_case("after", 991, [300, 17], num_q_heads=8, num_kv_heads=2, head_dim=128,
                                 block_size=16, dtype=torch.bfloat16)
    kc, vc = gpu_pools(case)
    ko, vo = oracle_pools(case)
    out = pa.paged_attention_decode(case.q.to(DEV), kc, vc, case.block_tables.to(DEV), case.seq_lens.to(DEV),
                                    case.scale)
    want = oracle.paged_attention_decode(case.q, ko, vo, case.block_tables, case.seq_lens, case.scale)
    check_close(out, want, torch.bfloat16, label="after timeout")


def test_selftest_refuses_bad_limits():
    lib = _lib.load()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert lib.pa_selftest_wait_timeout(0, err.data_ptr(), None) == _lib.PA_ERR_INVALID_ARGUMENT
    assert lib.pa_selftest_wait_timeout(10, None, None) == _lib.PA_ERR_INVALID_ARGUMENT
