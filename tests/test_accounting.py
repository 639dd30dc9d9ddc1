"""The bench's roofline accounting, pinned to the numbers "32. Production attention kernels"
prints (What the reference backend costs; The tests and the measurements)."""

import json
import os

import bench

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_bytes_qwen3_8b.json")


def test_bytes_per_token_matches_the_page():
    g = json.load(open(GOLDEN))
    per = bench.kv_bytes_per_token(g["num_kv_heads"], g["head_dim"], g["elem_bytes"])
    assert per == g["bytes_per_token_layer"] == 2 * g["values_per_token_layer"]
    assert per * g["num_layers"] == g["bytes_per_token_all_layers"]
    assert int(1e9 / g["bytes_per_token_all_layers"]) == g["tokens_per_GB"]


def test_decode_batch_bytes_and_floor_match_the_page():
    g = json.load(open(GOLDEN))
    b = g["batch"]
    kv = b["num_seqs"] * b["context"] * bench.kv_bytes_per_token(g["num_kv_heads"], g["head_dim"], g["elem_bytes"])
    assert kv == 1_073_741_824
    assert round(kv / 1e9, 2) == b["bytes_per_layer_GB"]
    assert round(kv * g["num_layers"] / 1e9, 1) == b["bytes_all_layers_GB"]
    assert round(kv * g["num_layers"] / (b["hbm_TBps"] * 1e12) * 1e3, 1) == b["floor_ms_all_layers"]
    # the decode call adds q, out and the used table entries on top of the cache itself
    call = bench.decode_call_bytes([4096] * 64, 32, 8, 128, 16, 2)
    assert call == kv + 2 * 64 * 32 * 128 * 2 + 64 * 256 * 4 + 64 * 4


def test_causal_flops():
    # full causal prompt of L: L(L+1)/2 visible pairs per head, 4*D flops each
    assert bench.causal_flops([8192] * 4, [8192] * 4, 32, 128) == 4.0 * 128 * 32 * 4 * 8192 * 8193 / 2
    # a chunk of 3 queries after 5 prior positions sees 6, 7, 8 keys
    assert bench.causal_flops([3], [8], 1, 1) == 4.0 * (6 + 7 + 8)
    assert bench.causal_flops([3], [8], 1, 1, causal=False) == 4.0 * 24
    # decode rows see their whole context
    assert bench.causal_flops([1, 1], [10, 20], 2, 4) == 4.0 * 4 * 2 * 30
