"""Oracle for the 8-bit KV cache: quantise on write, attend over the dequantised values.

Test infrastructure only (see the package docstring). Sources, by page title and section:

* "32. Production attention kernels", Quantized KV caches: one scale per (token, KV head),
  symmetric, scale = max|x| / q_max with q_max = 127 (int8) or 448 (fp8 E4M3), the largest
  element landing on the code range's edge; int8 codes are round(x / scale) clamped to
  [-127, 127], fp8 codes are x / scale cast to E4M3; the computation is in float32
  (``x.float()``); codes and scales are written through the same slot mapping as the
  values; the kernels dequantise the tile of codes by its per-slot scale.
* "TileInfer.jl - Attention kernels", INT8 cache: codes are exact in bf16 (|q| <= 127); a
  key's scale multiplies its row of scores and a value's scale its probability.

The attention itself is the float64 definition in ``attention.attend`` applied to
code * scale (both exact in float64).

Pins (tests/test_oracle_quant.py): the hand-derived golden quantisation and attention over
int8 / E4M3 codes (tests/golden/), the quantiser's error bound and range edge, a write/gather
round trip, and exact agreement (<= 1e-15) of both attention functions with the plain oracle
over a float64 pool of code * scale, with window, softcap and sinks; planted slips (swapped
key/value scales, a q_pos = t position rule, a shifted scale gather) fail them.
"""

from __future__ import annotations

import torch

from .attention import attend, default_scale

Q_MAX = {"int8": 127.0, "fp8": 448.0}
CODE_DTYPE = {"int8": torch.int8, "fp8": torch.float8_e4m3fn}


def quantize_kv(x: torch.Tensor, kind: str) -> tuple[torch.Tensor, torch.Tensor]:
    """x [N, Hkv, D] -> (codes [N, Hkv, D], scales [N, Hkv] float32), all arithmetic in float32.

    amax = max_d |x|, floored at 1e-8; scale = amax / q_max; codes = round-half-even(x / scale)
    clamped to +-127 (int8) or x / scale rounded to E4M3 (fp8)."""
    xf = x.to(torch.float32)
    amax = xf.abs().amax(dim=-1).clamp_min(1e-8)
    scale = amax / Q_MAX[kind]
    scaled = xf / scale[..., None]
    if kind == "int8":
        codes = scaled.round().clamp(-127, 127).to(torch.int8)
    else:
        codes = scaled.to(torch.float8_e4m3fn)
    return codes, scale


def reshape_and_cache_quant(key: torch.Tensor, value: torch.Tensor, k_codes: torch.Tensor, v_codes: torch.Tensor,
                            k_scales: torch.Tensor, v_scales: torch.Tensor, slot_mapping: torch.Tensor,
                            kind: str) -> None:
    """Quantise token rows and write codes and scales to slot ``slot_mapping[i]`` (-1 skips), in place.

    k_codes, v_codes: [num_blocks, block_size, Hkv, D]; k_scales, v_scales: [num_blocks, block_size, Hkv]."""
    kc, ks = quantize_kv(key, kind)
    vc, vs = quantize_kv(value, kind)
    block_size = k_codes.shape[1]
    capacity = k_codes.shape[0] * block_size
    for i in range(key.shape[0]):
        slot = int(slot_mapping[i])
        if slot < 0:
            continue
        if slot >= capacity:
            raise ValueError(f"slot {slot} outside a pool of {capacity} slots")
        b, o = slot // block_size, slot % block_size
        k_codes[b, o] = kc[i]
        v_codes[b, o] = vc[i]
        k_scales[b, o] = ks[i]
        v_scales[b, o] = vs[i]


def dequantized_context(codes: torch.Tensor, scales: torch.Tensor, table_row: torch.Tensor,
                        length: int) -> torch.Tensor:
    """Positions 0..length-1 of one sequence as code * scale in float64: [length, Hkv, D]."""
    block_size = codes.shape[1]
    if length == 0:
        return torch.zeros((0,) + tuple(codes.shape[2:]), dtype=torch.float64)
    n_pages = -(-length // block_size)
    pages = table_row[:n_pages].to(torch.long)
    c = codes.index_select(0, pages).reshape((n_pages * block_size,) + tuple(codes.shape[2:]))[:length]
    s = scales.index_select(0, pages).reshape((n_pages * block_size,) + tuple(scales.shape[2:]))[:length]
    return c.to(torch.float64) * s.to(torch.float64)[..., None]


def paged_attention_decode_quant(q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens,
                                 scale=None, seqs=None, window=0, softcap=0.0, sinks=None) -> torch.Tensor:
    """Decode over an 8-bit cache: the definition of oracle.paged_attention_decode on the
    dequantised keys and values."""
    S, Hq, D = q.shape
    sc = default_scale(D, scale)
    out = torch.zeros((S, Hq, D), dtype=torch.float64)
    for s in (range(S) if seqs is None else seqs):
        length = int(context_lens[s])
        keys = dequantized_context(k_codes, k_scales, block_tables[s], length)
        values = dequantized_context(v_codes, v_scales, block_tables[s], length)
        pos = torch.tensor([max(length - 1, 0)], dtype=torch.long)
        out[s] = attend(q[s:s + 1], pos, keys, values, sc, causal=False, window=window, softcap=softcap,
                        sinks=sinks)[0]
    return out


def paged_attention_varlen_quant(q, k_codes, v_codes, k_scales, v_scales, query_start_loc, seq_lens, block_tables,
                                 causal=True, scale=None, tokens=None, window=0, softcap=0.0,
                                 sinks=None) -> torch.Tensor:
    """Varlen attention over an 8-bit cache (positions as in oracle.paged_attention_varlen)."""
    N, Hq, D = q.shape
    sc = default_scale(D, scale)
    out = torch.zeros((N, Hq, D), dtype=torch.float64)
    wanted = None if tokens is None else set(int(t) for t in tokens)
    for r in range(seq_lens.shape[0]):
        start, stop = int(query_start_loc[r]), int(query_start_loc[r + 1])
        q_len, length = stop - start, int(seq_lens[r])
        if q_len < 0 or q_len > length:
            raise ValueError(f"request {r}: q_len {q_len} against seq_len {length}")
        rows = list(range(start, stop)) if wanted is None else [t for t in range(start, stop) if t in wanted]
        if not rows:
            continue
        keys = dequantized_context(k_codes, k_scales, block_tables[r], length)
        values = dequantized_context(v_codes, v_scales, block_tables[r], length)
        idx = torch.tensor(rows, dtype=torch.long)
        pos = length - q_len + (idx - start)
        out[idx] = attend(q.index_select(0, idx), pos, keys, values, sc, causal, window=window, softcap=softcap,
                          sinks=sinks)
    return out
