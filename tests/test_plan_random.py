"""The planner on seeded random batches (host only, no GPU).

The fixed workloads exercise the planner on a handful of shapes. Here each
seed draws a GQA configuration, a page size and a ragged batch that mixes
every kind of request the triple (q_start, q_end, kv_length) can state:
decodes, speculative multi-row decodes, chunks on top of a history, whole
prompts, and requests with no new rows. Some groups of requests map the same
physical pages for a leading part of their history (a shared prefix of any
length, not only the whole batch's), and the planner options are drawn too.
Every plan must cover each visible (row, head, key) exactly once, address
every key through a block-table row that holds the same pages there, give
split rows consecutive partial slots and skip no visible prefill tile (the
coverage check of ``test_abi``); no appended row may land in a page another
request maps.
"""

import math
import types

import numpy as np
import pytest

from continuous_batching_paged_varlen_gb300 import binding as B
from continuous_batching_paged_varlen_gb300 import build as build_mod
from tests.test_abi import check_coverage

HEADS = [(4, 4), (8, 2), (32, 8), (16, 2), (8, 8), (32, 32)]


@pytest.fixture(scope="module")
def L():
    build_mod.build()
    return B.lib()


def random_batch(seed, cap=None):
    """(workload-like namespace, plan options, shared groups) of one seed;
    ``cap`` bounds every kv_length (and so q_rows) for tests that also run
    the fp64 oracle."""
    rng = np.random.default_rng(seed)
    hq, hkv = HEADS[rng.integers(len(HEADS))]
    d = int(rng.choice([64, 128]))
    ps = int(rng.choice([16, 32, 64]))
    n = int(rng.integers(1, 13))
    shapes = []
    for _ in range(n):
        kind = rng.integers(5)
        if kind == 0:                      # decode
            kv = int(rng.integers(1, 3000))
            m = 1
        elif kind == 1:                    # speculative decode, k + 1 rows
            kv = int(rng.integers(5, 3000))
            m = int(rng.integers(2, 6))
        elif kind == 2:                    # chunk on top of a history
            m = int(rng.integers(1, 300))
            kv = m + int(rng.integers(0, 2000))
        elif kind == 3:                    # whole prompt, S0 = 0
            m = int(rng.integers(1, 600))
            kv = m
        else:                              # no new rows this iteration
            m = 0
            kv = int(rng.integers(0, 500))
        if cap is not None:
            kv = min(kv, cap)
            m = min(m, kv)
        shapes.append((m, kv))

    blocks = [math.ceil(kv / ps) for _, kv in shapes]
    max_blocks = max(max(blocks), 1)
    bt = np.full((n, max_blocks), -1, dtype=np.int32)
    # groups of 2-4 requests share the leading pages of their histories
    # (whole pages below every member's first new row: the append never
    # writes a shared page)
    order = rng.permutation(n)
    shared_of = {}
    i = 0
    while i < n:
        size = int(rng.integers(1, 5))
        members = [int(r) for r in order[i:i + size]]
        i += size
        if len(members) < 2 or rng.random() < 0.3:
            continue
        hist_pages = min((kv - m) // ps for m, kv in (shapes[r] for r in members))
        if hist_pages == 0:
            continue
        shared = int(rng.integers(1, hist_pages + 1))
        for r in members:
            shared_of[r] = (tuple(members), shared)
    n_pages = sum(blocks) + 7
    perm = rng.permutation(n_pages).astype(np.int32)
    cur = 0
    done = set()
    for r in range(n):
        start = 0
        if r in shared_of:
            members, shared = shared_of[r]
            if members not in done:
                ids = perm[cur:cur + shared]
                cur += shared
                for x in members:
                    bt[x, :shared] = ids
                done.add(members)
            start = shared
        bt[r, start:blocks[r]] = perm[cur:cur + blocks[r] - start]
        cur += blocks[r] - start
    assert cur <= n_pages

    reqs = np.zeros((n, 3), dtype=np.int32)
    q = 0
    for r, (m, kv) in enumerate(shapes):
        reqs[r] = (q, q + m, kv)
        q += m
    spec = types.SimpleNamespace(n_q_heads=hq, n_kv_heads=hkv, head_dim=d, page_size=ps,
                                 scale=None)
    w = types.SimpleNamespace(spec=spec, requests=reqs, block_table=bt, num_pages=n_pages,
                              total_q=q)

    choice = rng.integers(6)
    if choice == 0:
        opts = None
    elif choice == 1:
        opts = B.options(kv_chunk=64 * int(rng.integers(1, 9)))
    elif choice == 2:
        opts = B.options(prefill_min_rows=int(rng.choice([-1, 1, 16, 200])))
    elif choice == 3:
        opts = B.options(disable_cascade=1, kv_chunk=64 * int(rng.integers(1, 5)))
    elif choice == 4:
        opts = B.options(target_ctas=int(rng.choice([1, 7, 152, 1000])))
    else:
        opts = B.options(prefill_min_rows=int(rng.choice([-1, 0, 8])),
                         kv_chunk=64 * int(rng.integers(0, 4)),
                         disable_cascade=int(rng.integers(2)))
    return w, opts, shared_of


@pytest.mark.parametrize("seed", range(40))
def test_random_batches_are_covered_exactly_once(L, seed):
    w, opts, shared_of = random_batch(seed)
    hp, inf = check_coverage(w, opts)
    assert inf.total_q == w.total_q
    if opts is not None and opts.prefill_min_rows == -1:
        assert inf.n_prefill_items == 0
    if not shared_of or (opts is not None and opts.disable_cascade):
        assert inf.n_cascade_groups == 0
    cfg = B.config(w.spec.n_q_heads, w.spec.n_kv_heads, w.spec.head_dim, w.spec.page_size,
                   w.num_pages, w.block_table.shape[1])
    assert B.check_append_targets(w.requests, w.block_table, cfg) == (B.MB_OK, -1)
    hp.close()


def test_random_batches_use_every_kind_of_request_and_sharing(L):
    # the draw above reaches what it is meant to: shared groups, empty
    # requests, prefill items, split rows and cascade groups all occur
    seen = dict(shared=0, empty=0, prefill=0, combine=0, cascade=0)
    for seed in range(40):
        w, opts, shared_of = random_batch(seed)
        hp = B.HostPlan(w.requests, w.block_table, cfg_of(w), opts)
        inf = hp.info
        seen["shared"] += bool(shared_of)
        seen["empty"] += int(((w.requests[:, 1] - w.requests[:, 0]) == 0).any())
        seen["prefill"] += inf.n_prefill_items > 0
        seen["combine"] += inf.n_combine > 0
        seen["cascade"] += inf.n_cascade_groups > 0
        hp.close()
    assert all(v >= 3 for v in seen.values()), seen


def cfg_of(w):
    s = w.spec
    return B.config(s.n_q_heads, s.n_kv_heads, s.head_dim, s.page_size, w.num_pages,
                    w.block_table.shape[1])
