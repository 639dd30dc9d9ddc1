"""Seeded synthetic inputs for paged KV attention, shared by the tests and the bench.

This module only draws random numbers and lays them out as the library's
inputs (block tables, lengths, query rows, per-token keys/values and the slot
each token is written to). It holds none of the attention arithmetic, and it
imports neither the oracle nor the CUDA library.

Draw order for every case (torch.Generator on the CPU, seeded):
  1. lengths (randint, inclusive bounds), when the case draws them;
  2. randperm of the page pool;
  3. q, then k, then v, as float32 N(0, 1), cast to bf16 (round to nearest) for
     bf16 cases.
Pools start filled with NaN, so a kernel that reads an unused page or a tail
slot past a sequence's length shows it.

Named workloads (sizes from the hot path's published shapes: 32 query / 8 KV
heads of head_dim 128 is the Qwen3-8B attention shape the pages use):
  decode_1seq_fp32 / decode_ragged32_bf16 / decode_64x4096_bf16 (+ the
  head_dim 256 variant) / varlen_mixed_bf16 / prefill_4x8192_bf16 (+ head_dim 256
  and 64 variants).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


@dataclass
class PagedCase:
    """One synthetic batch. All tensors live on the CPU; move them as needed."""
    name: str
    dtype: torch.dtype
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    seq_lens: torch.Tensor            # [R] int32, positions cached including this step's tokens
    query_start_loc: torch.Tensor     # [R+1] int32
    block_tables: torch.Tensor        # [R, max_blocks] int32, zero padded
    q: torch.Tensor                   # [N, Hq, D]
    key: torch.Tensor                 # [T, Hkv, D] every cached token's key, request by request
    value: torch.Tensor               # [T, Hkv, D]
    slot_mapping: torch.Tensor        # [T] int32 pool slot of each row of key/value
    scale: float
    causal: bool = True
    meta: dict = field(default_factory=dict)

    @property
    def num_reqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_query_len(self) -> int:
        ql = self.query_start_loc[1:] - self.query_start_loc[:-1]
        return int(ql.max()) if ql.numel() else 0

    def empty_pools(self) -> tuple[torch.Tensor, torch.Tensor]:
        """NaN-filled [num_blocks, block_size, Hkv, D] key and value pools."""
        shape = (self.num_blocks, self.block_size, self.num_kv_heads, self.head_dim)
        return (torch.full(shape, float("nan"), dtype=self.dtype),
                torch.full(shape, float("nan"), dtype=self.dtype))


def _draw(gen: torch.Generator, shape, dtype: torch.dtype) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(dtype)


def make_case(name: str, seed: int, q_lens: list[int], seq_lens: list[int], *,
              num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
              dtype: torch.dtype, pool_blocks: int | None = None, table_multiple: int = 16,
              causal: bool = True, scale: float | None = None,
              gen: torch.Generator | None = None, meta: dict | None = None) -> PagedCase:
    """Lay out a batch of requests over a randomly permuted page pool.

    Request r holds seq_lens[r] cached positions (its q_lens[r] newest ones are
    this step's queries). Its pages take the next ids of a random permutation
    of the pool; the block table is zero padded to a multiple of
    ``table_multiple`` columns. ``pool_blocks`` defaults to exactly the pages
    needed.
    """
    if gen is None:
        gen = torch.Generator().manual_seed(seed)
    R = len(seq_lens)
    assert len(q_lens) == R
    pages = [cdiv(L, block_size) for L in seq_lens]
    need = sum(pages)
    num_blocks = max(need, 1) if pool_blocks is None else pool_blocks
    assert num_blocks >= need
    perm = torch.randperm(num_blocks, generator=gen).to(torch.int32)
    width = max(table_multiple, cdiv(max(pages + [1]), table_multiple) * table_multiple)
    tables = torch.zeros((R, width), dtype=torch.int32)
    cursor = 0
    for r in range(R):
        tables[r, :pages[r]] = perm[cursor:cursor + pages[r]]
        cursor += pages[r]
    qsl = torch.zeros(R + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int64), 0).to(torch.int32)
    n_tok = int(qsl[-1])
    total = sum(seq_lens)
    q = _draw(gen, (n_tok, num_q_heads, head_dim), dtype)
    key = _draw(gen, (total, num_kv_heads, head_dim), dtype)
    value = _draw(gen, (total, num_kv_heads, head_dim), dtype)
    # slot of every cached position, request by request, position by position
    slots = torch.empty(total, dtype=torch.int64)
    off = 0
    for r in range(R):
        L = seq_lens[r]
        pos = torch.arange(L, dtype=torch.int64)
        slots[off:off + L] = tables[r, pos // block_size].to(torch.int64) * block_size + pos % block_size
        off += L
    if scale is None:
        scale = head_dim ** -0.5
    return PagedCase(name=name, dtype=dtype, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                     head_dim=head_dim, block_size=block_size, num_blocks=num_blocks,
                     seq_lens=torch.tensor(seq_lens, dtype=torch.int32), query_start_loc=qsl,
                     block_tables=tables, q=q, key=key, value=value,
                     slot_mapping=slots.to(torch.int32), scale=float(scale), causal=causal,
                     meta=dict(meta or {}))


def decode_case(name: str, seed: int, context_lens: list[int], **kw) -> PagedCase:
    """A decode batch: one query per sequence (q_len 1 each)."""
    return make_case(name, seed, [1] * len(context_lens), context_lens, **kw)


# ---------------------------------------------------------------------------
# The named workloads of the hot path
# ---------------------------------------------------------------------------

def decode_1seq_fp32() -> PagedCase:
    """1 sequence, 200 cached positions (13 pages, last partial) in a pool of 32
    pages at permuted ids; 8 q heads over 2 KV heads, head_dim 64, block 16, fp32."""
    return decode_case("decode_1seq_fp32", 1001, [200], num_q_heads=8, num_kv_heads=2,
                       head_dim=64, block_size=16, dtype=torch.float32, pool_blocks=32)


def decode_ragged32_bf16() -> PagedCase:
    """32 sequences with lengths uniform in [1, 4096]; 32 q / 8 KV heads, head_dim
    128, block 16, bf16; pool = pages needed + 10% unused (rounded up)."""
    gen = torch.Generator().manual_seed(1002)
    lens = torch.randint(1, 4097, (32,), generator=gen).tolist()
    need = sum(cdiv(L, 16) for L in lens)
    return decode_case("decode_ragged32_bf16", 1002, lens, num_q_heads=32, num_kv_heads=8,
                       head_dim=128, block_size=16, dtype=torch.bfloat16,
                       pool_blocks=cdiv(need * 11, 10), gen=gen)


def decode_64x4096_bf16(head_dim: int = 128) -> PagedCase:
    """64 sequences x 4096 cached positions, block 16, bf16, pool exactly the
    16,384 pages needed, permuted. head_dim 128: 32 q / 8 KV heads; head_dim 256:
    16 q / 4 KV heads (the same 1,073,741,824 bytes of K+V)."""
    hq, hkv = (32, 8) if head_dim == 128 else (16, 4)
    name = "decode_64x4096_bf16" if head_dim == 128 else f"decode_64x4096_bf16_d{head_dim}"
    return decode_case(name, 1003 if head_dim == 128 else 1013,
                       [4096] * 64, num_q_heads=hq, num_kv_heads=hkv, head_dim=head_dim,
                       block_size=16, dtype=torch.bfloat16)


def varlen_mixed_bf16() -> PagedCase:
    """One flattened step: 8 prefill chunks of 512 new tokens (prior context
    uniform in [0, 2048]), 48 decode tokens (context uniform in [1, 4096]) and 8
    verify blocks of 5 tokens (context uniform in [1024, 4096]); 32 q / 8 KV
    heads, head_dim 128, block 16, bf16, causal."""
    gen = torch.Generator().manual_seed(1004)
    q_lens, seq_lens = [], []
    for _ in range(8):
        prior = int(torch.randint(0, 2049, (1,), generator=gen))
        q_lens.append(512)
        seq_lens.append(prior + 512)
    for _ in range(48):
        q_lens.append(1)
        seq_lens.append(int(torch.randint(1, 4097, (1,), generator=gen)))
    for _ in range(8):
        q_lens.append(5)
        seq_lens.append(int(torch.randint(1024, 4097, (1,), generator=gen)))
    return make_case("varlen_mixed_bf16", 1004, q_lens, seq_lens, num_q_heads=32,
                     num_kv_heads=8, head_dim=128, block_size=16, dtype=torch.bfloat16,
                     gen=gen)


def prefill_4x8192_bf16(head_dim: int = 128) -> PagedCase:
    """4 prompts of 8192 tokens each, causal, block 64 (512 permuted pages), bf16.
    head_dim 128: 32 q / 8 KV heads; head_dim 256: 16 q / 4 KV heads (the same causal flops);
    head_dim 64: 32 q / 8 KV heads."""
    if head_dim == 128:
        return make_case("prefill_4x8192_bf16", 1005, [8192] * 4, [8192] * 4, num_q_heads=32,
                         num_kv_heads=8, head_dim=128, block_size=64, dtype=torch.bfloat16)
    hq, hkv = (16, 4) if head_dim == 256 else (32, 8)
    return make_case(f"prefill_4x8192_bf16_d{head_dim}", 1015 if head_dim == 256 else 1016, [8192] * 4,
                     [8192] * 4, num_q_heads=hq, num_kv_heads=hkv, head_dim=head_dim, block_size=64,
                     dtype=torch.bfloat16)


def cascade_case(name: str, seed: int, prefix_len: int, suffix_lens: list[int], **kw) -> PagedCase:
    """S decode sequences behind one shared cached prefix: request 0 holds the prefix's
    prefix_len positions (no query), request 1 + s the s-th sequence's own suffix_lens[s]
    positions and its one query. The prefix's pages are block_tables[0]."""
    return make_case(name, seed, [0] + [1] * len(suffix_lens), [prefix_len] + list(suffix_lens), **kw)


def cascade_64x4000_bf16() -> PagedCase:
    """64 sequences sharing a 4,000-token prefix (250 pages of 16), each with its own suffix of
    1..256 positions (uniform); 32 q / 8 KV heads, head_dim 128, bf16."""
    gen = torch.Generator().manual_seed(1006)
    suffix = torch.randint(1, 257, (64,), generator=gen).tolist()
    return cascade_case("cascade_64x4000_bf16", 1006, 4000, suffix, num_q_heads=32, num_kv_heads=8,
                        head_dim=128, block_size=16, dtype=torch.bfloat16, gen=gen)


NAMED = {
    "decode_1seq_fp32": decode_1seq_fp32,
    "decode_ragged32_bf16": decode_ragged32_bf16,
    "decode_64x4096_bf16": decode_64x4096_bf16,
    "decode_64x4096_bf16_d256": lambda: decode_64x4096_bf16(256),
    "varlen_mixed_bf16": varlen_mixed_bf16,
    "prefill_4x8192_bf16": prefill_4x8192_bf16,
    "prefill_4x8192_bf16_d256": lambda: prefill_4x8192_bf16(256),
    "prefill_4x8192_bf16_d64": lambda: prefill_4x8192_bf16(64),
    "cascade_64x4000_bf16": cascade_64x4000_bf16,
}
