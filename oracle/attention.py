"""NumPy fp64 oracle for one attention step of a mixed continuous-batching
iteration over a paged, GQA KV cache.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

What is computed, and where the pages state it
----------------------------------------------
* Each request carries the triple ``(q_start, q_end, kv_length)``.
  ``q_rows = q_end - q_start`` new query rows; ``kv_length`` counts the whole
  context *after* this iteration's K/V have been appended.
  -- "ORCA and chunked prefill", section 2 (the per-request triple).
* With ``S0 = kv_length - q_rows`` cached positions and ``m = q_rows`` new
  ones, the first ``S0`` key columns are visible to every new row; among the
  last ``m`` columns only the strict upper triangle is masked (the diagonal
  stays visible). Masked scores are -inf before the softmax.
  -- "How To Scale Your Model notes (7-8)", section 2 (mask M); the same two
  blocks (unmasked prefix, lower-triangular chunk block) are described in
  "ORCA and chunked prefill", section 4.
* Scores are ``q . k * scale`` with ``scale = 1/sqrt(head_dim)`` unless
  overridden; the softmax subtracts the row maximum and each row of weights
  sums to one. -- "One forward, many requests" (batching many requests),
  section 6.2 (per-request loop, division by sqrt(d_head)); "LLM end to end",
  sections 4 and 6.
* Heads are independent; with GQA, ``g = Hq / Hkv`` query heads share one KV
  head, contiguously: query head ``h`` reads KV head ``h // g``.
  -- "LLM end to end", section 5; "How To Scale Your Model notes (7-8)",
  section 3 (GQA).
* K/V live in pages addressed through a per-request block table: logical
  position ``p`` is physical page ``block_table[p // page_size]``, slot
  ``p % page_size``. Paging changes only where data lives, never the result.
  -- "How To Scale Your Model notes (7-8)", section 3 (paging); "GLM-5.3
  e2e token ledger", stages 3 and 4 (64-token pages, block table,
  out_cache_loc).
* This iteration's K/V rows are appended to the cache before the attention
  reads it; new row ``t`` of a request sits at logical position
  ``S0 + (t - q_start)``. -- "ORCA and chunked prefill", section 4 (table:
  append K, V to the cache, then attention over S + C columns).

Physical cache layout used by the oracle's gather: ``[num_pages, Hkv,
page_size, D]`` for K and for V. The oracle addresses it with the formula
above, written out independently of the CUDA path.
"""

from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf


def default_scale(head_dim: int) -> float:
    """Softmax scale 1/sqrt(d_head) ("One forward, many requests", §6.2)."""
    return 1.0 / math.sqrt(head_dim)


def visible(s0: int, m: int) -> np.ndarray:
    """Visibility matrix ``[m, s0 + m]`` of the mask M.

    Row ``i`` (0-based new row) sees column ``j`` iff ``j < s0`` (cached
    history, always visible) or ``j - s0 <= i`` (own block, lower triangle
    including the diagonal). "How To Scale Your Model notes (7-8)", §2.
    """
    if s0 < 0 or m < 0:
        raise ValueError("s0 and m must be non-negative")
    vis = np.zeros((m, s0 + m), dtype=bool)
    vis[:, :s0] = True
    for i in range(m):
        vis[i, s0:s0 + i + 1] = True
    return vis


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float | None = None,
           return_weights: bool = False):
    """Attention of one request's new rows over its logical K/V.

    q: ``[m, Hq, D]``; k, v: ``[kv, Hkv, D]`` logical (gathered) history plus
    this iteration's rows, ``kv >= m``. Returns ``out [m, Hq, D]`` and
    ``lse [m, Hq]`` (natural log of the sum of exp of the visible scaled
    scores), both fp64; with ``return_weights`` also ``w [Hq, m, kv]``.
    The score matrix of each head is materialised and masked explicitly.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    m, hq, d = q.shape
    kv, hkv, dk = k.shape
    if dk != d or v.shape != k.shape:
        raise ValueError("q/k/v head dims disagree")
    if hq % hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    if m > kv:
        raise ValueError("q_rows must not exceed kv_length")
    g = hq // hkv
    if scale is None:
        scale = default_scale(d)
    s0 = kv - m
    vis = visible(s0, m)
    out = np.zeros((m, hq, d))
    lse = np.zeros((m, hq))
    weights = np.zeros((hq, m, kv)) if return_weights else None
    for h in range(hq):
        kh = h // g
        s = (q[:, h, :] @ k[:, kh, :].T) * scale          # [m, kv]
        s = np.where(vis, s, NEG_INF)
        row_max = s.max(axis=1, keepdims=True)             # finite: diagonal visible
        e = np.exp(s - row_max)                            # exp(-inf) = 0 on masked cells
        z = e.sum(axis=1, keepdims=True)
        w = e / z
        out[:, h, :] = w @ v[:, kh, :]
        lse[:, h] = row_max[:, 0] + np.log(z[:, 0])
        if return_weights:
            weights[h] = w
    if return_weights:
        return out, lse, weights
    return out, lse


def logical_position_location(block_table_row: np.ndarray, pos: int, page_size: int):
    """(physical page, slot) of logical position ``pos`` through a block table."""
    return int(block_table_row[pos // page_size]), pos % page_size


def gather_logical(cache: np.ndarray, block_table_row: np.ndarray, kv_length: int,
                   page_size: int) -> np.ndarray:
    """Logical ``[kv_length, Hkv, D]`` view of one request's paged K or V.

    ``cache`` is ``[num_pages, Hkv, page_size, D]``.
    """
    num_pages, hkv, ps, d = cache.shape
    if ps != page_size:
        raise ValueError("page_size disagrees with the cache layout")
    outv = np.empty((kv_length, hkv, d), dtype=cache.dtype)
    for p in range(kv_length):
        page, slot = logical_position_location(block_table_row, p, page_size)
        if not 0 <= page < num_pages:
            raise IndexError(f"block table entry {page} outside the page pool")
        outv[p] = cache[page, :, slot, :]
    return outv


def mixed_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                    requests, block_table: np.ndarray, page_size: int,
                    scale: float | None = None):
    """The whole attention step of one iteration (one layer).

    q: ``[total_q, Hq, D]`` flat over requests; caches ``[num_pages, Hkv,
    page_size, D]`` already holding this iteration's appended rows;
    ``requests``: rows of ``(q_start, q_end, kv_length)``; ``block_table``:
    ``[n_requests, max_blocks]``. Requests are walked one by one over their
    own slice of the flat tensor and their own pages only; cross-request
    blocks are never formed ("One forward, many requests", §6.2).
    Rows of ``q`` not covered by any request are left as zeros.
    """
    q = np.asarray(q, dtype=np.float64)
    total_q, hq, d = q.shape
    out = np.zeros((total_q, hq, d))
    lse = np.zeros((total_q, hq))
    for r, (q_start, q_end, kv_length) in enumerate(np.asarray(requests).tolist()):
        m = q_end - q_start
        if m == 0:
            continue
        k = gather_logical(k_cache, block_table[r], kv_length, page_size)
        v = gather_logical(v_cache, block_table[r], kv_length, page_size)
        o_r, l_r = attend(q[q_start:q_end], k, v, scale)
        out[q_start:q_end] = o_r
        lse[q_start:q_end] = l_r
    return out, lse


def append_scatter(k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray,
                   v_new: np.ndarray, requests, block_table: np.ndarray,
                   page_size: int):
    """KV append: write each new row into its page and slot, in place.

    Works on any dtype (the tests pass raw bf16 bit patterns as ``uint16`` so
    the comparison is bit-exact). New row ``t`` of request ``r`` goes to
    logical position ``p = S0 + (t - q_start)``, i.e. page
    ``block_table[r][p // page_size]``, slot ``p % page_size``.
    "ORCA and chunked prefill", §2 and §4; "GLM-5.3 e2e token ledger",
    stage 4 (out_cache_loc: which page and slot each new token goes to).
    """
    for r, (q_start, q_end, kv_length) in enumerate(np.asarray(requests).tolist()):
        m = q_end - q_start
        s0 = kv_length - m
        for t in range(q_start, q_end):
            p = s0 + (t - q_start)
            page, slot = logical_position_location(block_table[r], p, page_size)
            k_cache[page, :, slot, :] = k_new[t]
            v_cache[page, :, slot, :] = v_new[t]
    return k_cache, v_cache
