"""Host iteration builder (``include/mb_sched.h``), CPU only.

Every iteration of seeded random traces is checked against the rules the
builder follows ("ORCA and chunked prefill", sections 2-5; "GLM-5.3 e2e token
ledger", stage 3):

* the Q rows of an iteration fit its budget; decode steps have decode_rows
  rows; a prefill chunk never runs past the prompt;
* each triple's kv_length is the request's cached positions plus its rows;
* slots and positions agree with the library's own addressing helpers
  (``mb_slot_mapping``, ``mb_positions``, written independently);
* no page is held by two requests unless it is a shared prefix page, page
  reference counts add up, freed pages return to the pool;
* a prefix-cache hit reuses the cached pages (reference count + 1) and skips
  the prefix's recompute; page pressure preempts and the victims still finish.
"""

import numpy as np
import pytest

from continuous_batching_paged_varlen_gb300 import binding as B
from continuous_batching_paged_varlen_gb300 import build as build_mod


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_mod.build()
    B.lib()


def run_trace(sched, reqs, ps, max_steps=5000, check=True):
    """Drive ``sched`` until every request finished; check each iteration."""
    spec = {}
    for prompt, new, pid, plen in reqs:
        spec[sched.add(prompt, new, pid, plen)] = (prompt, new, pid, plen)
    history = []
    everyone = range(sched.n_added)  # requests queued before this call too
    for step in range(max_steps):
        before = {r: sched.request_info(r) for r in everyone}
        if all(i["state"] == "finished" for i in before.values()):
            break
        it = sched.step()
        if check:
            check_iteration(sched, it, before, ps)
        history.append((it, before))
        sched.commit()
        if it.total_q == 0:
            assert it.stats["n_running"] == 0 and it.stats["n_waiting"] == 0, \
                "empty iteration while requests wait"
    assert all(sched.request_info(r)["state"] == "finished" for r in everyone), \
        "trace did not finish"
    for r, (prompt, new, pid, plen) in spec.items():
        info = sched.request_info(r)
        assert info["state"] == "finished" and info["generated"] >= new and info["pages"] == 0
    return history


def check_iteration(sched, it, before, ps):
    cfg = sched.cfg
    n = len(it.ids)
    assert it.total_q <= cfg.token_budget
    # contiguous flat layout from row 0
    q = 0
    for k in range(n):
        qs, qe, kv = it.requests[k].tolist()
        assert qs == q and qe > qs
        q = qe
        info = before[int(it.ids[k])]
        rows = qe - qs
        if info["state"] == "decode":
            assert rows == cfg.decode_rows
        else:
            # prefill (or admission): never past the prompt; a prefix hit starts
            # at the cached prefix
            start = info["computed"] if info["state"] == "prefill" else kv - rows
            assert kv - rows == start and kv <= info["prompt_len"]
        if info["state"] != "waiting":
            assert kv - rows == info["computed"]
        # the block table covers every position up to kv_length
        bt = it.block_table[k]
        used = bt[bt >= 0]
        assert len(used) >= (kv + ps - 1) // ps
        assert len(set(used.tolist())) == len(used)
    assert q == it.total_q
    if n == 0:
        return
    # slots and positions by the library's own helpers
    ccfg = B.config(4, 4, 64, ps, cfg.num_pages, cfg.max_blocks_per_req)
    np.testing.assert_array_equal(it.slots, B.slot_mapping(it.requests, it.block_table, ccfg,
                                                           it.total_q))
    np.testing.assert_array_equal(it.positions, B.positions(it.requests, it.total_q))
    # the append contract: no new row lands in a page another request maps
    assert B.check_append_targets(it.requests, it.block_table, ccfg) == (B.MB_OK, -1)
    # pages: shared between requests only with a reference count to match
    refs = sched.page_refs()
    owners = {}
    for k in range(n):
        for p in it.block_table[k][it.block_table[k] >= 0].tolist():
            owners.setdefault(p, []).append(int(it.ids[k]))
            assert refs[p] >= 1
    for p, who in owners.items():
        assert refs[p] >= len(who)
        if len(who) > 1:
            pids = {before[r]["prefix_id"] for r in who}
            assert len(pids) == 1 and pids != {-1}, f"page {p} shared outside a prefix"
    assert int((refs == 0).sum()) == it.stats["free_pages"]


def test_short_trace_by_hand():
    s = B.Scheduler(num_pages=64, page_size=16, max_blocks_per_req=16, token_budget=48)
    a = s.add(100, 5)
    b = s.add(20, 3)
    it = s.step()
    assert it.requests.tolist() == [[0, 48, 48]] and it.ids.tolist() == [a]
    s.commit()
    it = s.step()
    assert it.requests.tolist() == [[0, 48, 96]]
    s.commit()
    it = s.step()  # the rest of a's prompt and all of b's in one iteration
    assert it.requests.tolist() == [[0, 4, 100], [4, 24, 20]] and it.ids.tolist() == [a, b]
    s.commit()
    it = s.step()  # two decode steps
    assert it.requests.tolist() == [[0, 1, 101], [1, 2, 21]]
    assert s.commit() == []
    s.step()
    assert s.commit() == [b]  # b's 1 + 2 outputs
    s.step()
    s.commit()
    s.step()
    assert s.commit() == [a]
    assert (s.page_refs() == 0).all()


def test_chunked_prefill_piggybacks_on_decodes():
    ps = 16
    s = B.Scheduler(num_pages=512, page_size=ps, max_blocks_per_req=128, token_budget=256)
    dec = [s.add(50, 200) for _ in range(8)]
    # let the decoders reach their decode phase
    while True:
        it = s.step()
        s.commit()
        if all(s.request_info(r)["state"] == "decode" for r in dec):
            break
    long = s.add(1500, 4)
    seen_chunks = []
    for _ in range(20):
        it = s.step()
        ids = it.ids.tolist()
        rows = {i: int(r[1] - r[0]) for i, r in zip(ids, it.requests)}
        if long in rows and s.request_info(long)["state"] != "decode":
            assert all(rows[d] == 1 for d in dec)  # every decoder keeps its step
            seen_chunks.append(rows[long])
        s.commit()
        if s.request_info(long)["state"] == "decode":
            break
    # chunks fill the budget left by the 8 decode rows, the last one the rest
    assert seen_chunks[:-1] == [256 - 8] * (len(seen_chunks) - 1)
    assert sum(seen_chunks) == 1500


@pytest.mark.parametrize("seed", range(8))
def test_random_traces_keep_the_invariants(seed):
    rng = np.random.default_rng(seed)
    ps = int(rng.choice([16, 32, 64]))
    n = int(rng.integers(3, 25))
    reqs = []
    for _ in range(n):
        prompt = int(rng.integers(1, 700))
        new = int(rng.integers(1, 60))
        if rng.random() < 0.3 and prompt > 2 * ps:
            pid = int(rng.integers(0, 3))
            reqs.append((prompt, new, pid, ps * int(rng.integers(1, prompt // ps))))
        else:
            reqs.append((prompt, new, -1, 0))
    max_ctx = max(p + k for p, k, _, _ in reqs)
    mb = (max_ctx + ps - 1) // ps + 1
    pool = int(rng.integers(mb + 1, 6 * mb))
    sched = B.Scheduler(num_pages=pool, page_size=ps, max_blocks_per_req=mb,
                        token_budget=int(rng.choice([64, 256, 1024])),
                        max_running=int(rng.choice([0, 4, 8])))
    run_trace(sched, reqs, ps)
    # at the end only prefix cache entries hold pages (one reference each)
    refs = sched.page_refs()
    assert refs.max() <= 1


def test_page_pressure_preempts_and_everyone_finishes():
    ps = 16
    sched = B.Scheduler(num_pages=24, page_size=ps, max_blocks_per_req=24, token_budget=512)
    reqs = [(60, 150, -1, 0) for _ in range(6)]
    hist = run_trace(sched, reqs, ps)
    assert sum(it.stats["n_preempted"] for it, _ in hist) > 0
    assert any(sched.request_info(r)["preemptions"] > 0 for r in range(6))
    assert (sched.page_refs() == 0).all()


def test_prefix_pages_are_shared_by_reference():
    ps, plen = 16, 64
    sched = B.Scheduler(num_pages=256, page_size=ps, max_blocks_per_req=32, token_budget=256)
    first = sched.add(100, 3, 7, plen)
    it = sched.step()
    first_pages = it.block_table[0][: plen // ps].tolist()
    sched.commit()
    while sched.request_info(first)["state"] != "decode":
        sched.step()
        sched.commit()
    others = [sched.add(80 + 10 * i, 5, 7, plen) for i in range(5)]
    it = sched.step()
    hits = it.stats["n_prefix_hits"]
    assert hits == 5
    refs = sched.page_refs()
    for k, rid in enumerate(it.ids.tolist()):
        if rid in others:
            qs, qe, kv = it.requests[k].tolist()
            assert kv - (qe - qs) == plen           # the prefix is not recomputed
            assert it.block_table[k][: plen // ps].tolist() == first_pages
    # users: the first request, the five new ones and the cache entry
    assert all(refs[p] == 7 for p in first_pages)
    sched.commit()
    run_trace(sched, [], ps)


def test_prefix_hit_needs_the_same_length():
    ps = 16
    sched = B.Scheduler(num_pages=128, page_size=ps, max_blocks_per_req=16, token_budget=512)
    sched.add(100, 2, 3, 64)
    sched.step()
    sched.commit()
    sched.add(100, 2, 3, 32)   # same id, shorter prefix: computes its own
    sched.add(120, 2, 3, 64)   # same id and length: hit
    it = sched.step()
    assert it.stats["n_prefix_hits"] == 1
    starts = {int(i): int(r[2] - (r[1] - r[0])) for i, r in zip(it.ids, it.requests)}
    assert starts[1] == 0 and starts[2] == 64
    sched.commit()
    run_trace(sched, [], ps)


def test_validation():
    with pytest.raises(B.MBError):
        B.Scheduler(num_pages=10, page_size=24, max_blocks_per_req=4, token_budget=8)
    s = B.Scheduler(num_pages=10, page_size=16, max_blocks_per_req=4, token_budget=8)
    with pytest.raises(B.MBError):
        s.add(0, 1)
    with pytest.raises(B.MBError):
        s.add(100, 1)  # 7 blocks > 4
    with pytest.raises(B.MBError):
        s.add(40, 1, 3, 20)  # prefix not page-aligned
    s.add(10, 1)
    s.step()
    with pytest.raises(B.MBError):
        s.step()  # the previous step is not committed
    s.commit()
    with pytest.raises(B.MBError):
        s.commit()
