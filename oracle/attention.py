"""The oracle: paged GQA attention written out as its definition, in float64.

Test infrastructure only (see the package docstring). Plain PyTorch CPU ops;
every floating-point step runs in float64 on values upcast exactly from the
stored bf16 / fp32 elements. Sources, by page title and section:

* "paged-attn-xpu", Method / Validation: the baseline gathers each sequence's
  pages into contiguous keys and values and runs a dense softmax in float64;
  an empty context gives zeros.
* "32. Production attention kernels", What the reference backend costs / One
  kernel for the whole batch: gather the request's blocks, repeat each KV head
  for its group of query heads, and place a request's q_len queries at the
  last q_len of its seq_len positions (query t sits at seq_len - q_len + t),
  causal by position.
* "poot - Attention and KV Cache", Attention as primitive ops / Multi-head,
  GQA, and MQA: scores = q.K^T * scale, max-subtracted softmax, times V; the
  KV head of query head h is h / n_rep.
* "poot - Attention and KV Cache", KV cache: new tokens are written through a
  write map of pool slots, -1 writing nothing.

Readings where the pages differ or are silent (each also listed in the design
notes): a row with no visible key returns zeros (the Triton chapter and
paged-attn-xpu; the poot page's 0/0 is not taken); ``scale`` of 0 or None means
1/sqrt(head_dim); slot s of the pool is row s % block_size of block
s // block_size.
"""

from __future__ import annotations

import math

import torch

_F64 = torch.float64


def default_scale(head_dim: int, scale: float | None) -> float:
    """Softmax scale: the caller's value, or 1/sqrt(head_dim) when it is 0/None.

    "32. Production attention kernels", One kernel for the whole batch (the
    launcher's ``scale or 1/sqrt(d)``); "paged-attn-xpu", Usage (scale=None).
    """
    if scale is None or scale == 0.0:
        return 1.0 / math.sqrt(head_dim)
    return float(scale)


def reshape_and_cache(key: torch.Tensor, value: torch.Tensor,
                      k_cache: torch.Tensor, v_cache: torch.Tensor,
                      slot_mapping: torch.Tensor) -> None:
    """Write token i's key/value rows into pool slot ``slot_mapping[i]``, in place.

    key, value: [N, Hkv, D]; k_cache, v_cache: [num_blocks, block_size, Hkv, D]
    of the same dtype; slot_mapping: [N] integers, -1 = write nothing.
    Slot s is (block s // block_size, row s % block_size).

    "poot - Attention and KV Cache", KV cache (write map, -1 skips);
    "32. Production attention kernels", Quantized KV caches (write_kv through
    the slot mapping, a plain copy of the bytes).
    """
    block_size = k_cache.shape[1]
    capacity = k_cache.shape[0] * block_size
    for i in range(key.shape[0]):
        slot = int(slot_mapping[i])
        if slot < 0:
            continue
        if slot >= capacity:
            raise ValueError(f"slot {slot} outside a pool of {capacity} slots")
        k_cache[slot // block_size, slot % block_size] = key[i]
        v_cache[slot // block_size, slot % block_size] = value[i]


def gather_context(cache: torch.Tensor, table_row: torch.Tensor, length: int) -> torch.Tensor:
    """Contiguous float64 copy of positions 0..length-1 of one sequence: [length, Hkv, D].

    Logical position p lives in page ``table_row[p // block_size]`` at row
    ``p % block_size``. The pages are fetched in table order, laid end to end,
    and cut to ``length`` ("paged-attn-xpu", Method; "32. Production attention
    kernels", What the reference backend costs, item 1).
    """
    block_size = cache.shape[1]
    if length == 0:
        return torch.zeros((0,) + tuple(cache.shape[2:]), dtype=_F64)
    n_pages = -(-length // block_size)
    pages = table_row[:n_pages].to(torch.long)
    if int(pages.min()) < 0 or int(pages.max()) >= cache.shape[0]:
        raise ValueError("block table names a page outside the pool")
    gathered = cache.index_select(0, pages)                    # [n_pages, bs, Hkv, D]
    flat = gathered.reshape((n_pages * block_size,) + tuple(cache.shape[2:]))
    return flat[:length].to(_F64)


def attend(q_rows: torch.Tensor, q_pos: torch.Tensor, keys: torch.Tensor,
           values: torch.Tensor, scale: float, causal: bool, window: int = 0,
           softcap: float = 0.0, sinks: torch.Tensor | None = None) -> torch.Tensor:
    """Masked softmax attention of some query rows over one sequence's keys.

    q_rows: [T, Hq, D]; q_pos: [T] positions of those queries; keys, values:
    [L, Hkv, D] (positions 0..L-1). Query head h reads KV head h // (Hq/Hkv).
    Key p is visible to a query at position t when p < L, if causal p <= t, and
    with a sliding window w > 0 also p > t - w ("32. Production attention
    kernels", One kernel for the whole batch: the window's extra mask term).
    Score s_p = scale * q.k_p, then, with a softcap c > 0, c * tanh(s_p / c)
    ("poot - Attention and KV Cache", The streaming schedule: softcap_or_identity).
    out[t, h] = sum_p e^{s_p} v_p / (e^{z_h} + sum_p e^{s_p}) over the visible p,
    where the optional sink logit z_h joins the denominator only ("32. Production
    attention kernels", Stretch exercises, attention sinks); without a sink the
    e^{z_h} term is absent. No visible key gives zeros. Returns [T, Hq, D] float64.
    """
    T, Hq, D = q_rows.shape
    L, Hkv, _ = keys.shape
    if Hq % Hkv != 0:
        raise ValueError("query heads must be a multiple of KV heads")
    group = Hq // Hkv
    q64 = q_rows.to(_F64)
    out = torch.zeros((T, Hq, D), dtype=_F64)
    if L == 0 or T == 0:
        return out
    key_pos = torch.arange(L, dtype=torch.long)
    pos = q_pos.to(torch.long)[:, None]
    if causal:
        visible = key_pos[None, :] <= pos                                     # [T, L]
    else:
        visible = torch.ones((T, L), dtype=torch.bool)
    if window > 0:
        visible = visible & (key_pos[None, :] > pos - window)
    any_visible = visible.any(dim=1)                                         # [T]
    neg_inf = torch.tensor(-math.inf, dtype=_F64)
    for h in range(Hq):
        kv = h // group
        scores = scale * (q64[:, h, :] @ keys[:, kv, :].T)                  # [T, L]
        if softcap > 0:
            scores = softcap * torch.tanh(scores / softcap)
        scores = torch.where(visible, scores, neg_inf)
        row_max = scores.max(dim=1, keepdim=True).values
        row_max = torch.where(any_visible[:, None], row_max, torch.zeros_like(row_max))
        if sinks is not None:
            z = float(sinks[h])
            row_max = torch.where(any_visible[:, None], torch.clamp(row_max, min=z), torch.full_like(row_max, z))
        weights = torch.where(visible, torch.exp(scores - row_max), torch.zeros_like(scores))
        denom = weights.sum(dim=1, keepdim=True)
        if sinks is not None:
            denom = denom + torch.exp(float(sinks[h]) - row_max)
        num = weights @ values[:, kv, :]                                     # [T, D]
        out[:, h, :] = torch.where(any_visible[:, None], num / torch.where(denom > 0, denom, 1.0),
                                   torch.zeros_like(num))
    return out


def paged_attention_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor,
                           scale: float | None = None,
                           seqs: list[int] | None = None, window: int = 0, softcap: float = 0.0,
                           sinks: torch.Tensor | None = None) -> torch.Tensor:
    """One query per sequence over its first ``context_lens[s]`` cached positions.

    q: [S, Hq, D]; caches [num_blocks, block_size, Hkv, D]; block_tables
    [S, max_blocks]; context_lens [S] (the length includes the query's own,
    already written, position). Returns [S, Hq, D] float64; rows of sequences
    not in ``seqs`` (when given) are left at zero.
    "paged-attn-xpu", Usage and Method; "32. Production attention kernels",
    Long contexts: split the keys (the exact result the splits must merge to).
    """
    S, Hq, D = q.shape
    sc = default_scale(D, scale)
    out = torch.zeros((S, Hq, D), dtype=_F64)
    for s in (range(S) if seqs is None else seqs):
        length = int(context_lens[s])
        if length < 0:
            raise ValueError("negative context length")
        keys = gather_context(k_cache, block_tables[s], length)
        values = gather_context(v_cache, block_tables[s], length)
        pos = torch.tensor([max(length - 1, 0)], dtype=torch.long)
        out[s] = attend(q[s:s + 1], pos, keys, values, sc, causal=False, window=window,
                        softcap=softcap, sinks=sinks)[0]
    return out


def paged_attention_varlen(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           query_start_loc: torch.Tensor, seq_lens: torch.Tensor,
                           block_tables: torch.Tensor, causal: bool = True,
                           scale: float | None = None,
                           tokens: torch.Tensor | None = None, window: int = 0,
                           softcap: float = 0.0, sinks: torch.Tensor | None = None) -> torch.Tensor:
    """A flattened batch: request r owns query rows query_start_loc[r]..[r+1]-1.

    Its q_len queries are the newest q_len of its seq_lens[r] positions: query
    t of request r sits at position seq_lens[r] - q_len + t, and sees key p
    when p < seq_lens[r] and (if causal) p <= its position ("32. Production
    attention kernels", One kernel for the whole batch, 'Points to notice').
    ``tokens`` (optional) restricts the evaluation to those flattened rows;
    the others stay zero. Returns [N, Hq, D] float64.
    """
    N, Hq, D = q.shape
    sc = default_scale(D, scale)
    out = torch.zeros((N, Hq, D), dtype=_F64)
    wanted = None if tokens is None else set(int(t) for t in tokens)
    R = seq_lens.shape[0]
    for r in range(R):
        start, stop = int(query_start_loc[r]), int(query_start_loc[r + 1])
        q_len = stop - start
        length = int(seq_lens[r])
        if q_len < 0 or q_len > length:
            raise ValueError(f"request {r}: q_len {q_len} against seq_len {length}")
        rows = list(range(start, stop)) if wanted is None else [t for t in range(start, stop) if t in wanted]
        if not rows:
            continue
        keys = gather_context(k_cache, block_tables[r], length)
        values = gather_context(v_cache, block_tables[r], length)
        idx = torch.tensor(rows, dtype=torch.long)
        pos = length - q_len + (idx - start)
        out[idx] = attend(q.index_select(0, idx), pos, keys, values, sc, causal, window=window,
                          softcap=softcap, sinks=sinks)
    return out


def cascade_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                   prefix_table: torch.Tensor, prefix_len: int, suffix_tables: torch.Tensor,
                   suffix_lens: torch.Tensor, scale: float | None = None) -> torch.Tensor:
    """Decode where every sequence's context is a shared prefix followed by its own suffix.

    Sequence s attends over prefix_len positions gathered from ``prefix_table`` and then
    suffix_lens[s] positions gathered from ``suffix_tables[s]``, laid end to end; its query is
    the last of them ("32. Production attention kernels", Long contexts: split the keys: the
    same merge serves cascade attention, a shared prefix attended once for many requests and
    merged with each request's own suffix). Returns [S, Hq, D] float64.
    """
    S, Hq, D = q.shape
    sc = default_scale(D, scale)
    out = torch.zeros((S, Hq, D), dtype=_F64)
    pk = gather_context(k_cache, prefix_table, prefix_len)
    pv = gather_context(v_cache, prefix_table, prefix_len)
    for s in range(S):
        length = int(suffix_lens[s])
        keys = torch.cat([pk, gather_context(k_cache, suffix_tables[s], length)], dim=0)
        values = torch.cat([pv, gather_context(v_cache, suffix_tables[s], length)], dim=0)
        total = keys.shape[0]
        pos = torch.tensor([max(total - 1, 0)], dtype=torch.long)
        out[s] = attend(q[s:s + 1], pos, keys, values, sc, causal=False)[0]
    return out
