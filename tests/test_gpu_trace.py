"""A multi-iteration serving trace through the whole library on the GPU.

The host iteration builder (``mb_sched_*``) schedules every iteration:
chunked prefills piggybacking on decode steps under a Q-row budget, a prefix
shared by reference between requests, and a KV pool small enough that pages
are preempted, freed and reused by other requests. Each iteration's new rows
go through ``mb_kv_append``, ``mb_attn_plan`` and ``mb_attn_forward``, and
every output row is compared with the fp64 oracle's attention over the
request's logical context -- so a page read that escapes its request, a stale
slot after reuse, or a wrong (q_start, q_end, kv_length) fails it.

Every (request, position) has fixed synthetic Q/K/V (the shared prefix's
K/V come from the prefix's own seed), so a preempted request recomputes the
same values when it is readmitted.
"""

import numpy as np
import pytest
import torch

from continuous_batching_paged_varlen_gb300 import binding as B
from oracle import attention as OA
from tests.gpu_harness import TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from continuous_batching_paged_varlen_gb300 import build
    build.build()
    B.lib()


def bf16_randn(gen, shape):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def make_values(reqs, hq, hkv, d, seed):
    """Per request: Q, K, V over its whole context [ctx, heads, d] (bf16, CPU).
    Requests sharing a prefix id get the prefix's K/V from the prefix seed."""
    prefix_kv = {}
    vals = []
    for r, (prompt, new, pid, plen) in enumerate(reqs):
        ctx = prompt + new
        g = torch.Generator().manual_seed(seed * 1000 + r)
        q = bf16_randn(g, (ctx, hq, d))
        k = bf16_randn(g, (ctx, hkv, d))
        v = bf16_randn(g, (ctx, hkv, d))
        if pid >= 0:
            if pid not in prefix_kv:
                gp = torch.Generator().manual_seed(seed * 1000 + 500 + pid)
                prefix_kv[pid] = (bf16_randn(gp, (plen, hkv, d)), bf16_randn(gp, (plen, hkv, d)))
            k[:plen], v[:plen] = prefix_kv[pid]
        vals.append((q, k, v))
    return vals


@pytest.mark.parametrize("hq,hkv,d,ps,pool,budget,new_max", [
    (4, 2, 64, 16, 28, 96, 40),     # tight pool: preemptions and page reuse
    (8, 2, 128, 32, 64, 256, 24),   # GQA 4, page 32
])
def test_scheduled_trace_matches_oracle(hq, hkv, d, ps, pool, budget, new_max):
    rng = np.random.default_rng(hq * 7 + d)
    reqs = [(int(rng.integers(10, 200)), int(rng.integers(2, new_max)), -1, 0) for _ in range(9)]
    reqs += [(150, 12, 0, 64), (200, 8, 0, 64), (90, 20, 0, 64)]  # a shared 64-position prefix
    max_ctx = max(p + n for p, n, _, _ in reqs)
    mb = (max_ctx + ps - 1) // ps + 1
    sched = B.Scheduler(num_pages=pool, page_size=ps, max_blocks_per_req=mb, token_budget=budget)
    for r in reqs:
        sched.add(*r)
    vals = make_values(reqs, hq, hkv, d, seed=hq + d)
    cfg = B.config(hq, hkv, d, ps, pool, mb)
    dev = "cuda"
    kc = torch.full((pool, hkv, ps, d), float("nan"), dtype=torch.bfloat16, device=dev)
    vc = torch.full((pool, hkv, ps, d), float("nan"), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    scale = 1.0 / np.sqrt(d)
    stats = {"iterations": 0, "preempted": 0, "prefix_hits": 0, "rows": 0}
    for _ in range(2000):
        it = sched.step()
        if it.total_q == 0:
            sched.commit()
            break
        stats["iterations"] += 1
        stats["preempted"] += it.stats["n_preempted"]
        stats["prefix_hits"] += it.stats["n_prefix_hits"]
        stats["rows"] += it.total_q
        # this iteration's new rows, in the flat layout of the triples
        rows_q, rows_k, rows_v = [], [], []
        for k_i, rid in enumerate(it.ids.tolist()):
            qs, qe, kv = it.requests[k_i].tolist()
            s0 = kv - (qe - qs)
            q, kk, vv = vals[rid]
            rows_q.append(q[s0:kv])
            rows_k.append(kk[s0:kv])
            rows_v.append(vv[s0:kv])
        q_flat = torch.cat(rows_q).to(dev)
        k_flat = torch.cat(rows_k).to(dev)
        v_flat = torch.cat(rows_v).to(dev)
        B.kv_append(kc, vc, k_flat, v_flat, torch.from_numpy(it.slots).to(dev), cfg, status)
        plan = B.Plan(it.requests, it.block_table, cfg, device=dev)
        out = torch.empty((it.total_q, hq, d), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((it.total_q, hq), dtype=torch.float32, device=dev)
        plan.forward(q_flat, kc, vc, torch.from_numpy(it.block_table).to(dev), out, lse)
        torch.cuda.synchronize()
        assert status.item() == 0 and plan.device_status() == 0
        plan.close()
        o_gpu = out.double().cpu().numpy()
        l_gpu = lse.double().cpu().numpy()
        for k_i, rid in enumerate(it.ids.tolist()):
            qs, qe, kv = it.requests[k_i].tolist()
            s0 = kv - (qe - qs)
            q, kk, vv = vals[rid]
            o_ref, l_ref = OA.attend(q[s0:kv].double().numpy(), kk[:kv].double().numpy(),
                                     vv[:kv].double().numpy(), scale)
            np.testing.assert_allclose(o_gpu[qs:qe], o_ref, rtol=TOL, atol=TOL,
                                       err_msg=f"request {rid} rows {s0}:{kv}")
            np.testing.assert_allclose(l_gpu[qs:qe], l_ref, rtol=TOL, atol=TOL)
        sched.commit()
    assert all(sched.request_info(r)["state"] == "finished" for r in range(len(reqs)))
    assert stats["prefix_hits"] >= 1
    if pool == 28:
        assert stats["preempted"] >= 1
