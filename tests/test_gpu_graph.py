"""An iteration's launches captured once in a CUDA graph and replayed.

A serving loop builds each iteration's inputs into static buffers so that
the forward can be replayed as a captured CUDA graph instead of launching
each kernel from the host ("GLM-5.3 e2e token ledger", stage 4: the input
batch, its slot mapping and block table, CUDA-graph buffers). This file
captures ``mb_kv_append`` + ``mb_attn_forward`` (the plan is made and
uploaded beforehand, outside the capture), then writes new Q / K / V values
into the static input buffers before each replay and checks every replay
against the fp64 oracle. Replays must start clean: the split-KV kernel's
per-row arrival counters go back to zero inside the kernel, and the
workspace status word stays 0.
"""

import dataclasses

import numpy as np
import pytest
import torch

from continuous_batching_paged_varlen_gb300 import binding as B
from continuous_batching_paged_varlen_gb300 import workloads as W
from tests.gpu_harness import assert_request_close, cfg_of, poisoned_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from continuous_batching_paged_varlen_gb300 import build
    build.build()
    B.lib()


def _history(w, kc, vc, cfg):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    n_hist = int(w.hist_requests[:, 1].max()) if len(w.hist_requests) else 0
    if n_hist:
        slots = B.slot_mapping(w.hist_requests, w.block_table, cfg, n_hist)
        B.kv_append(kc, vc, w.k_hist.cuda(), w.v_hist.cuda(), torch.from_numpy(slots).cuda(),
                    cfg, status)
    torch.cuda.synchronize()
    assert status.item() == 0


def _fresh_values(w, seed):
    g = torch.Generator().manual_seed(seed)

    def rnd(t):
        return torch.randn(t.shape, generator=g).to(torch.bfloat16)

    return dataclasses.replace(w, q=rnd(w.q), k_new=rnd(w.k_new), v_new=rnd(w.v_new))


@pytest.mark.parametrize("name,opts", [("tiny_mixed", dict(kv_chunk=64)),
                                       ("shared_prefix_decode", None)])
def test_captured_iteration_replays_match_the_oracle(name, opts):
    w = W.make_workload(name)
    cfg = cfg_of(w)
    s = w.spec
    kc, vc = poisoned_cache(w, "cuda")
    _history(w, kc, vc, cfg)
    o = B.options(**opts) if opts else None
    plan = B.Plan(w.requests, w.block_table, cfg, device="cuda", opts=o)
    if opts:
        assert plan.info.n_combine > 0  # split rows: the in-kernel merge runs every replay

    # static buffers the graph is captured over
    q = w.q.cuda()
    k_new, v_new = w.k_new.cuda(), w.v_new.cuda()
    slots = torch.from_numpy(B.slot_mapping(w.requests, w.block_table, cfg, w.total_q)).cuda()
    bt = torch.from_numpy(np.ascontiguousarray(w.block_table)).cuda()
    out = torch.zeros((w.total_q, s.n_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((w.total_q, s.n_q_heads), dtype=torch.float32, device="cuda")
    ast = torch.zeros(1, dtype=torch.int32, device="cuda")

    def iteration():
        B.kv_append(kc, vc, k_new, v_new, slots, cfg, ast)
        plan.forward(q, kc, vc, bt, out, lse)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # first launches (per-device set-up) outside the capture
        iteration()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        iteration()
    torch.cuda.synchronize()

    for replay, seed in enumerate((101, 202, 303)):
        wr = _fresh_values(w, seed)
        q.copy_(wr.q)
        k_new.copy_(wr.k_new)
        v_new.copy_(wr.v_new)
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert ast.item() == 0
        assert plan.device_status() == 0, f"replay {replay}"
        for r in range(len(w.requests)):
            assert_request_close(wr, out, lse, r)
    graph.reset()
    plan.close()


def test_captured_fp8_iteration_replays_match_the_oracle():
    """The same on the fp8 cache: the quantizing append of this iteration's
    rows and the split-KV forward over the codes (shared-prefix cascade, split
    rows merged in the kernel), captured once and replayed with new values."""
    from tests.test_gpu_fp8 import check_all, empty_caches, slots_of

    w = W.make_workload("shared_prefix_decode")
    cfg = cfg_of(w)
    s = w.spec
    ps = s.page_size
    k8, v8, ks, vs = empty_caches(w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    hs = torch.from_numpy(slots_of(w.hist_requests, w.block_table, ps).astype(np.int32)).cuda()
    B.kv_append_fp8(k8, v8, ks, vs, w.k_hist.cuda(), w.v_hist.cuda(), hs, cfg, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    plan = B.Plan(w.requests, w.block_table, cfg, device="cuda",
                  opts=B.options(prefill_min_rows=-1))
    assert plan.info.n_combine > 0 and plan.info.n_cascade_groups == 1

    q = w.q.cuda()
    k_new, v_new = w.k_new.cuda(), w.v_new.cuda()
    slots = torch.from_numpy(slots_of(w.requests, w.block_table, ps).astype(np.int32)).cuda()
    bt = torch.from_numpy(np.ascontiguousarray(w.block_table)).cuda()
    out = torch.zeros((w.total_q, s.n_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((w.total_q, s.n_q_heads), dtype=torch.float32, device="cuda")

    def iteration():
        B.kv_append_fp8(k8, v8, ks, vs, k_new, v_new, slots, cfg, st)
        plan.forward_fp8(q, k8, v8, ks, vs, bt, out, lse)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        iteration()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        iteration()
    torch.cuda.synchronize()

    for replay, seed in enumerate((404, 505)):
        wr = _fresh_values(w, seed)
        q.copy_(wr.q)
        k_new.copy_(wr.k_new)
        v_new.copy_(wr.v_new)
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert st.item() == 0
        assert plan.device_status() == 0, f"replay {replay}"
        check_all(wr, out, lse)
    graph.reset()
    plan.close()
