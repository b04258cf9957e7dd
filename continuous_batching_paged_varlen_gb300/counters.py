"""Algorithmic work counters for the attention step (bench bookkeeping).

These count what the method must do, not what a kernel happens to do:

* FLOPs: ``4 * D`` per (query head, visible (q, k) pair) -- a multiply-add for
  each of the ``D`` products in ``q.k`` and in ``w.v``. Per request
  ``pairs = q_rows * S0 + q_rows (q_rows + 1) / 2`` (unmasked prefix block
  plus the lower triangle of the own block). Masked-out pairs never count.
  Over a whole network this is ``4 * d_head * heads * layers`` per pair,
  "ORCA and chunked prefill", §3 (the Llama-2-7B cost model, ~0.52 MFLOP).
* HBM bytes: Q read + O write (bf16) + every *distinct* physical K/V position
  the step reads, once (``2 * Hkv * D * 2`` bytes per position, K and V) +
  the block-table entries. Positions whose pages are shared by several
  requests count once: a per-position KV size ``2 * layers * Hkv * D * 2``
  gives the 128 KiB of "How To Scale Your Model notes (7-8)", §3, and six
  requests sharing a 4096-position prefix plus 1024 private positions read
  3.75 GiB naively against 1.25 GiB stored.
* Append bytes: read the new K/V rows and write them into their slots.
"""

from __future__ import annotations

import numpy as np


def bytes_per_position(n_layers: int, n_kv_heads: int, head_dim: int,
                       elem_bytes: int = 2) -> int:
    """K and V bytes one token position occupies across all layers."""
    return 2 * n_layers * n_kv_heads * head_dim * elem_bytes


def flops_per_pair(head_dim: int, n_heads: int, n_layers: int = 1) -> int:
    """Attention FLOPs of one visible (q, k) pair over heads and layers."""
    return 4 * head_dim * n_heads * n_layers


def pairs(q_rows: int, kv_length: int) -> int:
    s0 = kv_length - q_rows
    return q_rows * s0 + q_rows * (q_rows + 1) // 2


def attention_flops(requests, n_q_heads: int, head_dim: int) -> int:
    tot = 0
    for qs, qe, kv in np.asarray(requests).tolist():
        tot += pairs(qe - qs, kv)
    return tot * flops_per_pair(head_dim, n_q_heads)


def distinct_kv_positions(requests, block_table, page_size: int) -> int:
    """Distinct physical (page, slot) positions the step reads."""
    seen = {}
    for r, (qs, qe, kv) in enumerate(np.asarray(requests).tolist()):
        nb = (kv + page_size - 1) // page_size
        for b in range(nb):
            page = int(block_table[r][b])
            filled = min(page_size, kv - b * page_size)
            seen[page] = max(seen.get(page, 0), filled)
    return int(sum(seen.values()))


def naive_kv_positions(requests) -> int:
    """K/V positions read when every request scans its own history."""
    return int(sum(kv for _, _, kv in np.asarray(requests).tolist()))


def attention_bytes(requests, block_table, n_q_heads: int, n_kv_heads: int,
                    head_dim: int, page_size: int, elem_bytes: int = 2,
                    kv_elem_bytes: int | None = None, kv_row_scale_bytes: int = 0) -> int:
    """kv_elem_bytes: bytes per cached K/V value (default elem_bytes; 1 for
    the fp8 cache); kv_row_scale_bytes: per (position, KV head) scale bytes of
    K and of V (4 for the fp8 cache's fp32 scales)."""
    reqs = np.asarray(requests)
    total_q = int((reqs[:, 1] - reqs[:, 0]).sum())
    qo = 2 * total_q * n_q_heads * head_dim * elem_bytes
    kvb = elem_bytes if kv_elem_bytes is None else kv_elem_bytes
    kv = (distinct_kv_positions(reqs, block_table, page_size) * 2 * n_kv_heads
          * (head_dim * kvb + kv_row_scale_bytes))
    bt = int(sum((kv_len + page_size - 1) // page_size for _, _, kv_len in reqs.tolist())) * 4
    return qo + kv + bt


def append_bytes(n_new_tokens: int, n_kv_heads: int, head_dim: int,
                 elem_bytes: int = 2) -> int:
    """Read the new K and V rows and write them into the cache, + slots."""
    return 2 * 2 * n_new_tokens * n_kv_heads * head_dim * elem_bytes + 4 * n_new_tokens


def rope_append_bytes(n_new_tokens: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                      elem_bytes: int = 2) -> int:
    """Fused rotary embedding + append: read and write every query row (rotated
    in place), read K and V and write them into the cache, read the token's
    angle-table row (fp32) and its position and slot."""
    per_token = (2 * n_q_heads * head_dim * elem_bytes + 4 * n_kv_heads * head_dim * elem_bytes
                 + head_dim * 4 + 8)
    return n_new_tokens * per_token


def append_fp8_bytes(n_new_tokens: int, n_kv_heads: int, head_dim: int) -> int:
    """Quantizing append: read the new bf16 K and V rows, write their e4m3
    codes and one fp32 scale per (token, KV head) row of each, + slots."""
    return n_new_tokens * (2 * n_kv_heads * (head_dim * 2 + head_dim + 4) + 4)
