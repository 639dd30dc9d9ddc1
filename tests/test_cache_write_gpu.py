"""pa_reshape_and_cache is a copy: bit-exact against the oracle's scatter."""

import pytest
import torch

import oracle
import paged_kv_attention_gb300 as pa
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("hkv,d,bs", [(8, 128, 16), (4, 256, 64), (2, 64, 1), (1, 64, 128)])
def test_bit_exact_with_padding_slots(dtype, hkv, d, bs):
    case = workloads.make_case("w", 5 + d + bs, [1, 1, 1], [37, 300, 5], num_q_heads=hkv, num_kv_heads=hkv,
                               head_dim=d, block_size=bs, dtype=dtype, pool_blocks=None)
    slots = case.slot_mapping.clone()
    slots[::7] = -1                                         # padding tokens write nothing
    kc, vc = (t.to(DEV) for t in case.empty_pools())
    pa.reshape_and_cache(case.key.to(DEV), case.value.to(DEV), kc, vc, slots.to(DEV))
    ko, vo = case.empty_pools()
    oracle.reshape_and_cache(case.key, case.value, ko, vo, slots)
    torch.cuda.synchronize()
    assert torch.equal(_bits(kc.cpu()), _bits(ko))
    assert torch.equal(_bits(vc.cpu()), _bits(vo))


def test_prefill_sized_write_is_bit_exact():
    case = workloads.prefill_4x8192_bf16()
    kc, vc = (t.to(DEV) for t in case.empty_pools())
    pa.reshape_and_cache(case.key.to(DEV), case.value.to(DEV), kc, vc, case.slot_mapping.to(DEV))
    ko, vo = case.empty_pools()
    # same scatter on the CPU, vectorised through the oracle's own slot rule via index_copy of rows
    oracle.reshape_and_cache(case.key[:64], case.value[:64], ko, vo, case.slot_mapping[:64])
    bs = case.block_size
    flat_k = kc.cpu().view(-1, case.num_kv_heads, case.head_dim)
    slots = case.slot_mapping.long()
    assert torch.equal(_bits(flat_k[slots]), _bits(case.key))
    flat_v = vc.cpu().view(-1, case.num_kv_heads, case.head_dim)
    assert torch.equal(_bits(flat_v[slots]), _bits(case.value))
    # the first 64 tokens also agree with the oracle's scatter, slot for slot
    first = slots[:64]
    assert torch.equal(_bits(kc.cpu()[first // bs, first % bs]), _bits(ko[first // bs, first % bs]))


def test_out_of_pool_slot_is_skipped_and_flagged():
    case = workloads.make_case("bad", 9, [1], [20], num_q_heads=2, num_kv_heads=2, head_dim=128, block_size=16,
                               dtype=torch.bfloat16)
    slots = case.slot_mapping.clone()
    slots[3] = case.num_blocks * 16 + 100
    slots[4] = -7
    kc, vc = (t.to(DEV) for t in case.empty_pools())
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.reshape_and_cache(case.key.to(DEV), case.value.to(DEV), kc, vc, slots.to(DEV), error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa._lib.PA_ERRBIT_SLOT_OUT_OF_POOL
    ko, vo = case.empty_pools()
    good = slots.clone()
    good[3] = -1
    good[4] = -1
    oracle.reshape_and_cache(case.key, case.value, ko, vo, good)
    assert torch.equal(_bits(kc.cpu()), _bits(ko))
