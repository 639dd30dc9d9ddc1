"""Host planner of the tensor-core varlen grid (pa_varlen_plan): the items it lists are exactly
the (query tile pair, request) pairs the batch has, each once, longest first; short requests are
left out when the call will serve them with the split-KV decode. No GPU needed."""

import pytest
import torch

import paged_kv_attention_gb300 as pa

from test_abi import lib  # noqa: F401  (builds the library if stale)


def key_tiles(q_len, seq, tok0, tok, causal, window):
    n = max(0, min(tok, q_len - tok0))
    if n == 0:
        return 0
    first = seq - q_len + tok0
    end = min(seq, first + n) if causal else seq
    j0 = max(0, first - window + 1) // 128 if window > 0 else 0
    return max(0, -(-max(0, end) // 128) - j0)


@pytest.mark.parametrize("hq,hkv", [(32, 8), (16, 1), (8, 8)])
@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 300)])
@pytest.mark.parametrize("split", [False, True])
def test_plan_lists_each_existing_pair_once_longest_first(lib, hq, hkv, causal, window, split):  # noqa: F811
    q_lens = [512, 1, 5, 0, 37, 130, 8, 9, 64, 1, 300]
    seq_lens = [2048, 4000, 900, 3, 37, 900, 8, 100, 64, 1, 3000]
    qsl = torch.zeros(len(q_lens) + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(torch.tensor(q_lens), 0)
    sl = torch.tensor(seq_lens, dtype=torch.int32)
    g = hq // hkv
    tok = 128 // g
    items = pa.varlen_plan(qsl, sl, max(q_lens), hq, hkv, causal, window, split_decodes=split)
    r_count = len(q_lens)
    got = [(int(i) // r_count, int(i) % r_count) for i in items]
    want = {(t, r) for r, ql in enumerate(q_lens) if ql > 0 and not (split and ql <= 8)
            for t in range(-(-ql // (2 * tok)))}
    assert len(got) == len(set(got)) == len(want)
    assert set(got) == want
    work = [max(key_tiles(q_lens[r], seq_lens[r], t * 2 * tok, tok, causal, window),
                key_tiles(q_lens[r], seq_lens[r], t * 2 * tok + tok, tok, causal, window)) for t, r in got]
    assert all(a >= b for a, b in zip(work, work[1:]))


def test_plan_refuses_small_capacity_and_bad_arguments(lib):  # noqa: F811
    qsl = torch.tensor([0, 300, 301], dtype=torch.int32)
    sl = torch.tensor([300, 50], dtype=torch.int32)
    out = torch.zeros(64, dtype=torch.int32)
    n = lib.pa_varlen_plan(qsl.data_ptr(), sl.data_ptr(), 2, 300, 32, 8, 1, 0, 0, out.data_ptr(), 64)
    assert n == 6  # 300 tokens in pairs of 64, plus the one-token request
    assert lib.pa_varlen_plan(qsl.data_ptr(), sl.data_ptr(), 2, 300, 32, 8, 1, 0, 0, out.data_ptr(), 5) == -1
    assert lib.pa_varlen_plan(qsl.data_ptr(), sl.data_ptr(), 2, 300, 32, 6, 1, 0, 0, out.data_ptr(), 64) == -1
    assert lib.pa_varlen_plan_capacity(2, 300, 32, 8) == 10
    assert lib.pa_varlen_plan_capacity(2, 300, 64, 2) == -1   # group 32
    assert lib.pa_varlen_plan(qsl.data_ptr(), sl.data_ptr(), 0, 300, 32, 8, 1, 0, 0, out.data_ptr(), 0) == 0
