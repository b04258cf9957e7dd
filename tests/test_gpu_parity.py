"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Caches are filled with NaN before the appends, so a kernel that reads an
unwritten slot (or lets one reach the output through a zero weight) fails.
Cache writes must be bit-exact; outputs and LSEs within atol = rtol = 2e-2.
"""

import numpy as np
import pytest
import torch

from continuous_batching_paged_varlen_gb300 import binding as B
from continuous_batching_paged_varlen_gb300 import workloads as W
from oracle import attention as OA
from tests.gpu_harness import (TOL, assert_request_close, cfg_of, custom_workload, fill_cache,
                               run_forward)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from continuous_batching_paged_varlen_gb300 import build
    build.build()
    B.lib()


# ------------------------------------------------------------------ append

def oracle_cache_bits(w):
    s = w.spec
    kc = np.full((w.num_pages, s.n_kv_heads, s.page_size, s.head_dim), 0x7FC0, np.uint16)
    vc = kc.copy()
    as_bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)  # noqa: E731
    OA.append_scatter(kc, vc, as_bits(w.k_hist), as_bits(w.v_hist), w.hist_requests,
                      w.block_table, s.page_size)
    OA.append_scatter(kc, vc, as_bits(w.k_new), as_bits(w.v_new), w.requests, w.block_table,
                      s.page_size)
    return kc, vc


@pytest.mark.parametrize("name", ["tiny_mixed", "llama2_7b_orca_iteration",
                                  "shared_prefix_decode"])
def test_append_bit_exact(name):
    w = W.make_workload(name)
    kc, vc, _ = fill_cache(w)
    ok, ov = oracle_cache_bits(w)
    gk = kc.view(torch.int16).cpu().numpy().view(np.uint16)
    gv = vc.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(gk, ok)
    assert np.array_equal(gv, ov)


def test_append_padding_and_bad_slot_flag():
    w = W.make_workload("tiny_mixed")
    cfg = cfg_of(w)
    s = w.spec
    kc = torch.zeros((w.num_pages, s.n_kv_heads, s.page_size, s.head_dim), dtype=torch.bfloat16,
                     device="cuda")
    vc = torch.zeros_like(kc)
    kn = torch.randn(3, s.n_kv_heads, s.head_dim, device="cuda").to(torch.bfloat16)
    vn = torch.randn(3, s.n_kv_heads, s.head_dim, device="cuda").to(torch.bfloat16)
    slots = torch.tensor([5, -1, w.num_pages * s.page_size + 7], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.kv_append(kc, vc, kn, vn, slots, cfg, status)
    torch.cuda.synchronize()
    assert status.item() == 1 << B.MB_ERR_DEVICE_INDEX
    assert torch.equal(kc[0, :, 5], kn[0]) and torch.equal(vc[0, :, 5], vn[0])
    assert int((kc.float().abs().sum(dim=(1, 3)).cpu() != 0).sum()) == 1
    # T = 0 enqueues nothing
    B.kv_append(kc, vc, kn, vn, slots[:0], cfg, status)


# --------------------------------------------------------------- attention

OPTION_SETS = {
    "default": None,
    "all_split_kv": dict(prefill_min_rows=-1),
    "all_prefill": dict(prefill_min_rows=1),
    "chunk64": dict(kv_chunk=64),
    "chunk256_nocascade": dict(kv_chunk=256, disable_cascade=1),
}


@pytest.mark.parametrize("opt", sorted(OPTION_SETS))
def test_tiny_mixed_parity(opt):
    w = W.make_workload("tiny_mixed")
    kc, vc, cfg = fill_cache(w)
    o = OPTION_SETS[opt]
    out, lse, status, info = run_forward(w, kc, vc, cfg, B.options(**o) if o else None)
    assert status == 0
    for r in range(w.n_requests):
        assert_request_close(w, out, lse, r)


def test_llama_iteration_parity_sampled():
    w = W.make_workload("llama2_7b_orca_iteration")
    kc, vc, cfg = fill_cache(w)
    out, lse, status, info = run_forward(w, kc, vc, cfg)
    assert status == 0 and info["n_prefill_items"] == 32 * 16
    assert torch.isfinite(out.float()).all()
    # the 4096-row prefill: three heads in full (every tile, ragged-free)
    assert_request_close(w, out, lse, 0, heads=[0, 13, 31])
    # the two decodes: every head
    assert_request_close(w, out, lse, 1)
    assert_request_close(w, out, lse, 2)


def test_decode_heavy_parity_sampled():
    w = W.make_workload("decode_heavy_gqa4", device="cuda")
    kc, vc, cfg = fill_cache(w)
    out, lse, status, info = run_forward(w, kc, vc, cfg)
    assert status == 0
    assert torch.isfinite(out.float()).all()
    rng = np.random.default_rng(0)
    for r in sorted(rng.choice(w.n_requests, 12, replace=False).tolist()) + [0, w.n_requests - 1]:
        assert_request_close(w, out, lse, r)


def test_chunked_prefill_mix_parity_sampled():
    w = W.make_workload("chunked_prefill_mix", device="cuda")
    kc, vc, cfg = fill_cache(w)
    out, lse, status, info = run_forward(w, kc, vc, cfg)
    assert status == 0
    assert torch.isfinite(out.float()).all()
    # the 2048-row chunk at S0 = 30720: first, middle and last rows, two heads
    for rows in [(0, 48), (1000, 1040), (2000, 2048)]:
        assert_request_close(w, out, lse, 0, heads=[0, 29], rows=rows)
    for r in [1, 17, 40, 64]:
        assert_request_close(w, out, lse, r)


def test_spec_decode_parity_sampled():
    # k + 1 = 4 new rows per request: causal among the step's own rows
    w = W.make_workload("spec_decode_k3", device="cuda")
    kc, vc, cfg = fill_cache(w)
    out, lse, status, info = run_forward(w, kc, vc, cfg)
    assert status == 0 and info["n_prefill_items"] == 0
    assert torch.isfinite(out.float()).all()
    rng = np.random.default_rng(1)
    for r in sorted(rng.choice(w.n_requests, 8, replace=False).tolist()) + [0, w.n_requests - 1]:
        assert_request_close(w, out, lse, r)


def test_varlen_prefill_parity_sampled():
    # prefill-only ragged batch (S0 = 0 everywhere): each request's own causal
    # block only, never a cross-request block
    w = W.make_workload("varlen_prefill", device="cuda")
    kc, vc, cfg = fill_cache(w)
    out, lse, status, info = run_forward(w, kc, vc, cfg)
    assert status == 0 and info["n_decode_items"] == 0
    assert torch.isfinite(out.float()).all()
    for r in [0, 5, 11, w.n_requests - 1]:
        m = int(w.requests[r, 1] - w.requests[r, 0])
        for a, b in [(0, 40), (m // 2 - 20, m // 2 + 20), (m - 40, m)]:
            assert_request_close(w, out, lse, r, heads=[0, 17, 31], rows=(a, b))


@pytest.mark.parametrize("cascade", [True, False])
def test_shared_prefix_parity(cascade):
    w = W.make_workload("shared_prefix_decode", device="cuda")
    kc, vc, cfg = fill_cache(w)
    out, lse, status, info = run_forward(
        w, kc, vc, cfg, None if cascade else B.options(disable_cascade=1))
    assert status == 0
    assert info["n_cascade_groups"] == (1 if cascade else 0)
    for r in range(6):
        assert_request_close(w, out, lse, r)


EDGE_CASES = {
    # name: (shapes, kwargs)
    "q0_and_kv1": ([(0, 5), (1, 1), (3, 3), (1, 17)], {}),
    "ragged_tiles_tail": ([(129, 300), (255, 255), (1, 77)], dict(n_q_heads=4, n_kv_heads=1)),
    "page32_d128_g8": ([(40, 700), (1, 33), (2, 65)],
                       dict(n_q_heads=16, n_kv_heads=2, head_dim=128, page_size=32)),
    "page128_mha": ([(200, 1000), (1, 129), (16, 16)],
                    dict(n_q_heads=2, n_kv_heads=2, head_dim=128, page_size=128)),
    "page64_shared_pairs": ([(1, 600), (1, 700), (2, 650)],
                            dict(n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=64,
                                 shared_prefix=512)),
    "scale_override": ([(33, 90), (1, 50)], dict(scale=0.05)),
}


@pytest.mark.parametrize("case", sorted(EDGE_CASES))
@pytest.mark.parametrize("opt", ["default", "all_split_kv", "all_prefill"])
def test_edge_cases(case, opt):
    shapes, kw = EDGE_CASES[case]
    w = custom_workload(shapes, seed=sum(map(ord, case)), **kw)
    kc, vc, cfg = fill_cache(w)
    o = OPTION_SETS[opt]
    out, lse, status, info = run_forward(w, kc, vc, cfg, B.options(**o) if o else None)
    assert status == 0
    for r in range(w.n_requests):
        if w.requests[r, 1] > w.requests[r, 0]:
            assert_request_close(w, out, lse, r)


def test_a_thousand_short_requests():
    # the most requests of any test: 1000 requests of every kind but long
    # (decodes at kv 1..300, 4-row speculative steps, 24-row chunks), so the
    # plan has thousands of short split-KV CTAs and prefill items; every
    # request checked in full
    rng = np.random.default_rng(33)
    shapes = [(1, 1), (1, 16)]
    for i in range(998):
        kind = i % 3
        if kind == 0:
            shapes.append((1, int(rng.integers(1, 301))))
        elif kind == 1:
            shapes.append((4, int(rng.integers(4, 301))))
        else:
            shapes.append((24, int(rng.integers(24, 301))))
    w = custom_workload(shapes, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=16, seed=33)
    kc, vc, cfg = fill_cache(w)
    out, lse, status, info = run_forward(w, kc, vc, cfg)
    assert status == 0 and info["n_prefill_items"] > 0 and info["n_decode_items"] > 600
    for r in range(w.n_requests):
        assert_request_close(w, out, lse, r)


def test_long_context_many_partials():
    # the largest ranges of any test: a 131072-key decode (with a 1024-key
    # chunk: 128 partials per row, which the in-kernel merge reads 16 slots
    # at a time), a 65537-key decode, and a 300-row chunk over a 100k-key
    # history (sampled rows and heads); the default plan and the forced split
    w = custom_workload([(1, 131072), (300, 100000), (1, 65537)], n_q_heads=8, n_kv_heads=2,
                        head_dim=128, page_size=64, seed=21)
    kc, vc, cfg = fill_cache(w)
    for opts in (None, B.options(kv_chunk=1024)):
        out, lse, status, info = run_forward(w, kc, vc, cfg, opts)
        assert status == 0
        if opts is not None:
            assert info["n_partials"] >= 128 * 8 + 65 * 8
        assert_request_close(w, out, lse, 0)
        assert_request_close(w, out, lse, 2)
        for rows in [(0, 16), (284, 300)]:
            assert_request_close(w, out, lse, 1, heads=[0, 5], rows=rows)


# Long key ranges (>= 8 tiles of 128 keys per split-KV CTA). A plan with
# most of its keys in such CTAs of <= 32 rows runs the split-KV build that
# spreads each row's keys over 4 copies in the softmax warps; its CTAs with
# more rows or short ranges keep one thread per row. Cases: copies alone,
# with partials, a shared-prefix group, and mixed with a 40-row CTA; plans
# that stay on the other build.
COPY_CASES = {
    # (shapes, workload kw, planner options, split-KV build expected)
    "4_rows_copies": ([(1, 5000), (1, 2600)], dict(n_q_heads=8, n_kv_heads=2, head_dim=128,
                                                   page_size=64), dict(kv_chunk=8192), 1),
    "split_rows_copies": ([(1, 9000), (2, 7000)], dict(n_q_heads=8, n_kv_heads=2,
                                                       head_dim=128, page_size=64),
                          dict(kv_chunk=2560), 1),
    "cascade_32_rows_copies": ([(1, 4200 + 13 * i) for i in range(8)],
                               dict(n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=64,
                                    shared_prefix=4096), dict(kv_chunk=4096), 1),
    "copies_with_a_40_row_cta": ([(1, 6000), (10, 5000), (1, 7000)],
                                 dict(n_q_heads=8, n_kv_heads=2, head_dim=64, page_size=32),
                                 dict(kv_chunk=8192, prefill_min_rows=-1), 1),
    "1_row_ctas_of_10_to_15_tiles_copies": ([(1, 1200), (1, 1900), (1, 1500)],
                                            dict(n_q_heads=4, n_kv_heads=4, head_dim=128,
                                                 page_size=16), dict(kv_chunk=2048), 1),
    "short_ranges_one_per_thread": ([(1, 600), (1, 500), (2, 520)],
                                    dict(n_q_heads=8, n_kv_heads=2, head_dim=128,
                                         page_size=64), dict(kv_chunk=1024), 0),
    "48_rows_one_per_thread": ([(12, 4000)], dict(n_q_heads=8, n_kv_heads=2, head_dim=128,
                                                  page_size=64),
                               dict(kv_chunk=8192, prefill_min_rows=-1), 0),
    "100_rows_one_per_thread": ([(25, 3000)], dict(n_q_heads=8, n_kv_heads=2, head_dim=64,
                                                   page_size=32),
                                dict(kv_chunk=8192, prefill_min_rows=-1), 0),
}


@pytest.mark.parametrize("case", sorted(COPY_CASES))
def test_long_ranges_split_kv_builds(case):
    shapes, kw, opts, build = COPY_CASES[case]
    w = custom_workload(shapes, seed=sum(map(ord, case)), **kw)
    kc, vc, cfg = fill_cache(w)
    out, lse, status, info = run_forward(w, kc, vc, cfg, B.options(**opts))
    assert status == 0
    assert info["splitkv_copies"] == build
    if "cascade" in case:
        assert info["n_cascade_groups"] == 1
    for r in range(w.n_requests):
        assert_request_close(w, out, lse, r)


def test_deterministic_and_empty():
    w = W.make_workload("tiny_mixed")
    kc, vc, cfg = fill_cache(w)
    a = run_forward(w, kc, vc, cfg)[0]
    b = run_forward(w, kc, vc, cfg)[0]
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    empty = custom_workload([])
    plan = B.Plan(empty.requests, np.zeros((0, 1), np.int32), cfg_of(empty))
    assert plan.info.n_launches == 0
    plan.forward(None, None, None, None, None)
    plan.close()


@pytest.mark.parametrize("name,opts", [("tiny_mixed", dict(kv_chunk=64)),
                                       ("shared_prefix_decode", {}),
                                       ("spec_decode_k3", dict(kv_chunk=256))])
def test_split_rows_merged_on_every_forward(name, opts):
    """Split rows are merged by the CTA that completes them, through per-row
    arrival counters that each merge puts back to zero: the same plan run
    again (and again) must give the same, complete rows."""
    if name == "spec_decode_k3":  # a bounded share of the batch
        sp = W.SPECS[name]
        w = custom_workload(W.request_shapes(sp)[:24], n_q_heads=sp.n_q_heads,
                            n_kv_heads=sp.n_kv_heads, head_dim=sp.head_dim,
                            page_size=sp.page_size, seed=5)
    else:
        w = W.make_workload(name)
    kc, vc, cfg = fill_cache(w)
    plan = B.Plan(w.requests, w.block_table, cfg, opts=B.options(**opts))
    assert plan.info.n_combine > 0 and plan.info.n_launches == 1 + (plan.info.n_prefill_items > 0)
    s = w.spec
    q = w.q.cuda()
    bt = torch.from_numpy(np.ascontiguousarray(w.block_table)).cuda()
    results = []
    for _ in range(3):
        out = torch.full((w.total_q, s.n_q_heads, s.head_dim), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        lse = torch.full((w.total_q, s.n_q_heads), float("nan"), dtype=torch.float32,
                         device="cuda")
        plan.forward(q, kc, vc, bt, out, lse)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        results.append((out, lse))
    plan.close()
    for out, lse in results[1:]:
        assert torch.equal(out.view(torch.int16), results[0][0].view(torch.int16))
        assert torch.equal(lse.view(torch.int32), results[0][1].view(torch.int32))
    out, lse = results[0]
    for r in range(w.n_requests):
        if w.requests[r, 1] > w.requests[r, 0]:
            assert_request_close(w, out, lse, r, heads=range(0, s.n_q_heads, 7))


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    """Failure path shared by every kernel's waits: a wait on an mbarrier that
    nothing completes gives up after its limit (2 s), flags MB_ERR_TIMEOUT in
    the status word and the kernel returns; the next forward runs normally."""
    import time
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    B.selftest_wait_timeout(status)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(status.item()) == 1 << B.MB_ERR_TIMEOUT
    assert 1.5 < waited < 30.0
    w = W.make_workload("tiny_mixed")
    kc, vc, cfg = fill_cache(w)
    out, lse, st, _ = run_forward(w, kc, vc, cfg)
    assert st == 0
    for r in range(w.n_requests):
        if w.requests[r, 1] > w.requests[r, 0]:
            assert_request_close(w, out, lse, r)
