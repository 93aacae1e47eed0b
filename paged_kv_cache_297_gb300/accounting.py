"""Algorithmic byte and flop counts used for roofline fractions.

These are measurement formulas, not part of the computed path.  The KV bytes
follow the ledger of chengxuchu PyTorch #47, section 2.3
(layers x 2 x batch x kv_heads x sequence_length x head_dim x bytes) and the
per-request form on caffein.top, "KV Cache is the hard constraint"
(2 x layers x tokens x kv_heads x head_dim x bytes), evaluated for one layer
and each sequence's own context length.
"""

from __future__ import annotations

import torch

BLOCK_SIZE = 16


def kv_cache_bytes(layers: int, batch: int, kv_heads: int, seq_len: int, head_dim: int,
                   bytes_per_element: int) -> int:
    """Size of a dense KV cache (K and V)."""
    return layers * 2 * batch * kv_heads * seq_len * head_dim * bytes_per_element


def decode_bytes(context_lens: torch.Tensor, num_q_heads: int, num_kv_heads: int,
                 head_dim: int, elem: int, out_elem: int, q_elem: int | None = None) -> dict:
    """Bytes one decode launch must move at minimum.

    KV: every cached token of every sequence, K and V, each kv head once
    (``elem`` bytes per cached element: 1 for an fp8 cache).  Plus the query
    (``q_elem``, default ``elem``) and output rows, each sequence's used
    block-table entries and its context length.  Split-K partials are
    overhead and not counted.
    """
    q_elem = elem if q_elem is None else q_elem
    L = context_lens.to(torch.int64)
    tokens = int(L.sum())
    kv = kv_cache_bytes(1, 1, num_kv_heads, tokens, head_dim, elem)
    S = int(L.numel())
    qo = S * num_q_heads * head_dim * (q_elem + out_elem)
    tables = int(((L + BLOCK_SIZE - 1) // BLOCK_SIZE).sum()) * 4 + S * 4
    return {"kv": kv, "q_out": qo, "tables": tables, "total": kv + qo + tables}


def append_bytes(num_tokens: int, num_kv_heads: int, head_dim: int, elem: int) -> int:
    """K and V rows read once and written once, plus the slot ids."""
    return 2 * 2 * num_tokens * num_kv_heads * head_dim * elem + 8 * num_tokens


def copy_blocks_bytes(num_pairs: int, num_kv_heads: int, head_dim: int, elem: int) -> int:
    """Each pair reads and writes one whole K block and one whole V block."""
    return num_pairs * 2 * 2 * num_kv_heads * BLOCK_SIZE * head_dim * elem + 16 * num_pairs


def causal_pairs(prior: int, n: int) -> int:
    """(query, key) pairs of a chunk of n queries after ``prior`` cached tokens:
    query j sees prior + j + 1 keys."""
    return n * prior + n * (n + 1) // 2


def prefill_flops(cu_q_lens: torch.Tensor, context_lens: torch.Tensor, num_q_heads: int,
                  head_dim: int) -> int:
    """2*d flops for q.k plus 2*d for p.v per causal (query, key) pair and head;
    the masked-out upper triangle is not counted."""
    cu = cu_q_lens.to(torch.int64).tolist()
    L = context_lens.to(torch.int64).tolist()
    pairs = 0
    for s in range(len(L)):
        n = cu[s + 1] - cu[s]
        pairs += causal_pairs(L[s] - n, n)
    return 4 * head_dim * num_q_heads * pairs
