"""Helpers shared by the GPU parity tests: build paged caches through the
library's append, run the forward, and compute the oracle on the same seeded
inputs (copied to the host)."""

from __future__ import annotations

import math

import numpy as np
import torch

from continuous_batching_paged_varlen_gb300 import binding as B
from continuous_batching_paged_varlen_gb300 import workloads as W
from oracle import attention as OA

TOL = 2e-2  # atol = rtol, on bf16 outputs with fp32 accumulation
BF16_NAN = 0x7FC0


def cfg_of(w) -> B.Config:
    s = w.spec
    return B.config(s.n_q_heads, s.n_kv_heads, s.head_dim, s.page_size, w.num_pages,
                    w.block_table.shape[1], s.scale or 0.0)


def poisoned_cache(w, device, poison=True):
    s = w.spec
    shape = (w.num_pages, s.n_kv_heads, s.page_size, s.head_dim)
    if poison:
        c = torch.full(shape, BF16_NAN, dtype=torch.int16, device=device).view(torch.bfloat16)
        d = torch.full(shape, BF16_NAN, dtype=torch.int16, device=device).view(torch.bfloat16)
        return c, d
    return (torch.zeros(shape, dtype=torch.bfloat16, device=device),
            torch.zeros(shape, dtype=torch.bfloat16, device=device))


def fill_cache(w, device="cuda", poison=True):
    """History rows then this iteration's rows, both through mb_kv_append."""
    cfg = cfg_of(w)
    kc, vc = poisoned_cache(w, device, poison)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    n_hist = int(w.hist_requests[:, 1].max()) if len(w.hist_requests) else 0
    if n_hist:
        hslots = B.slot_mapping(w.hist_requests, w.block_table, cfg, n_hist)
        B.kv_append(kc, vc, w.k_hist.to(device), w.v_hist.to(device),
                    torch.from_numpy(hslots).to(device), cfg, status)
    slots = B.slot_mapping(w.requests, w.block_table, cfg, w.total_q)
    B.kv_append(kc, vc, w.k_new.to(device), w.v_new.to(device),
                torch.from_numpy(slots).to(device), cfg, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return kc, vc, cfg


def run_forward(w, kc, vc, cfg, opts=None, device="cuda", with_lse=True):
    plan = B.Plan(w.requests, w.block_table, cfg, device=device, opts=opts)
    s = w.spec
    q = w.q.to(device)
    out = torch.full((w.total_q, s.n_q_heads, s.head_dim), float("nan"), dtype=torch.bfloat16,
                     device=device)
    lse = torch.full((w.total_q, s.n_q_heads), float("nan"), dtype=torch.float32,
                     device=device) if with_lse else None
    bt_dev = torch.from_numpy(np.ascontiguousarray(w.block_table)).to(device)
    plan.forward(q, kc, vc, bt_dev, out, lse)
    torch.cuda.synchronize()
    status = plan.device_status()
    info = plan.info.as_dict()
    plan.close()
    return out, lse, status, info


def oracle_request(w, r, heads=None, rows=None):
    """fp64 oracle output/LSE of request r (optionally a subset of query heads
    and a contiguous subset [a, b) of its new rows)."""
    qs, qe, kv = [int(x) for x in w.requests[r]]
    m = qe - qs
    s0 = kv - m
    a, b = (0, m) if rows is None else rows
    k, v = w.logical_kv(r)
    k = k[: s0 + b].to(torch.float64).cpu().numpy()
    v = v[: s0 + b].to(torch.float64).cpu().numpy()
    q = w.q[qs + a: qs + b].to(torch.float64).cpu().numpy()
    spec = w.spec
    g = spec.n_q_heads // spec.n_kv_heads
    heads = list(range(spec.n_q_heads)) if heads is None else list(heads)
    outs, lses = [], []
    for h in heads:
        kh = h // g
        o, l = OA.attend(q[:, h:h + 1], k[:, kh:kh + 1], v[:, kh:kh + 1], spec.scale)
        outs.append(o[:, 0])
        lses.append(l[:, 0])
    return np.stack(outs, 1), np.stack(lses, 1), (qs + a, qs + b), heads


def assert_request_close(w, out, lse, r, heads=None, rows=None, tol=TOL):
    o_ref, l_ref, (t0, t1), heads = oracle_request(w, r, heads, rows)
    o_gpu = out[t0:t1][:, heads].to(torch.float64).cpu().numpy()
    assert np.isfinite(o_gpu).all(), f"non-finite output in request {r}"
    np.testing.assert_allclose(o_gpu, o_ref, rtol=tol, atol=tol,
                               err_msg=f"request {r} rows {t0}:{t1}")
    if lse is not None:
        l_gpu = lse[t0:t1][:, heads].to(torch.float64).cpu().numpy()
        np.testing.assert_allclose(l_gpu, l_ref, rtol=tol, atol=tol,
                                   err_msg=f"lse request {r}")


def custom_workload(shapes, n_q_heads=4, n_kv_heads=2, head_dim=64, page_size=16, seed=0,
                    shared_prefix=0, pool_extra=3, scale=None):
    spec = W.WorkloadSpec(name="custom", n_q_heads=n_q_heads, n_kv_heads=n_kv_heads,
                          head_dim=head_dim, page_size=page_size, requests=tuple(shapes),
                          shared_prefix=shared_prefix, seed=seed, scale=scale)
    blocks = sum(math.ceil(kv / page_size) for _, kv in shapes) if shapes else 1
    spec = W.WorkloadSpec(**{**spec.__dict__, "pool_pages": blocks + pool_extra})
    return W.make_workload(spec)
