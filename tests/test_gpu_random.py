"""Seeded random batches through the CUDA path, against the fp64 oracle.

The batches of ``test_plan_random`` (every kind of request, shared prefixes
of any length among groups of requests, random planner options), with kv
lengths capped so that the oracle runs in about a second: every page of the
pool holds seeded N(0,1) bf16 values, this iteration's rows are appended by
``mb_kv_append`` on the GPU and by the oracle's scatter on the host, and the
whole step (``mixed_attention``: per request, gather through the block table,
masked softmax in fp64) is compared with ``mb_attn_forward`` on every row and
head. Cache writes must be bit-exact.

The same batches on the fp8 (e4m3) cache: every slot of the pool is written
through the quantizing append, then this iteration's rows; codes and scales
must equal the oracle's bit for bit, and ``mb_attn_forward_fp8`` (split-KV
work lists only) must match ``mixed_attention`` over the K/V the oracle
dequantized itself.
"""

import numpy as np
import pytest
import torch

from continuous_batching_paged_varlen_gb300 import binding as B
from oracle import attention as OA
from oracle import fp8 as F
from tests.gpu_harness import TOL
from tests.test_plan_random import cfg_of, random_batch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from continuous_batching_paged_varlen_gb300 import build
    build.build()
    B.lib()


@pytest.mark.parametrize("seed", range(24))
def test_random_batch_matches_the_oracle(seed):
    w, opts, _ = random_batch(seed, cap=800)
    s = w.spec
    cfg = cfg_of(w)
    gen = torch.Generator().manual_seed(10_000 + seed)
    shape = (w.num_pages, s.n_kv_heads, s.page_size, s.head_dim)
    kc = torch.randn(shape, generator=gen).to(torch.bfloat16)
    vc = torch.randn(shape, generator=gen).to(torch.bfloat16)
    q = torch.randn((w.total_q, s.n_q_heads, s.head_dim), generator=gen).to(torch.bfloat16)
    kn = torch.randn((w.total_q, s.n_kv_heads, s.head_dim), generator=gen).to(torch.bfloat16)
    vn = torch.randn((w.total_q, s.n_kv_heads, s.head_dim), generator=gen).to(torch.bfloat16)

    # oracle: the host copy of the pool, this iteration's rows scattered in
    hk, hv = kc.float().numpy(), vc.float().numpy()
    OA.append_scatter(hk, hv, kn.float().numpy(), vn.float().numpy(), w.requests,
                      w.block_table, s.page_size)
    o_ref, l_ref = OA.mixed_attention(q.float().numpy(), hk, hv, w.requests, w.block_table,
                                      s.page_size)

    dkc, dvc = kc.cuda(), vc.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if w.total_q:
        slots = torch.from_numpy(B.slot_mapping(w.requests, w.block_table, cfg, w.total_q))
        B.kv_append(dkc, dvc, kn.cuda(), vn.cuda(), slots.cuda(), cfg, status)
    plan = B.Plan(w.requests, w.block_table, cfg, device="cuda", opts=opts)
    out = torch.full((max(w.total_q, 1), s.n_q_heads, s.head_dim), float("nan"),
                     dtype=torch.bfloat16, device="cuda")
    lse = torch.full((max(w.total_q, 1), s.n_q_heads), float("nan"), device="cuda")
    bt = torch.from_numpy(np.ascontiguousarray(w.block_table)).cuda()
    plan.forward(q.cuda() if w.total_q else out, dkc, dvc, bt, out, lse)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert plan.device_status() == 0
    plan.close()

    # cache writes bit-exact (the whole pool: untouched pages stay as they were)
    ref_k = torch.from_numpy(hk).to(torch.bfloat16)
    ref_v = torch.from_numpy(hv).to(torch.bfloat16)
    assert torch.equal(dkc.cpu().view(torch.int16), ref_k.view(torch.int16))
    assert torch.equal(dvc.cpu().view(torch.int16), ref_v.view(torch.int16))

    rows = np.zeros(max(w.total_q, 1), dtype=bool)
    for qs, qe, _ in w.requests.tolist():
        rows[qs:qe] = True
    if not rows.any():
        return
    got = out.double().cpu().numpy()[rows]
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, o_ref[rows[:w.total_q]], rtol=TOL, atol=TOL,
                               err_msg=f"seed {seed}")
    np.testing.assert_allclose(lse.double().cpu().numpy()[rows], l_ref[rows[:w.total_q]],
                               rtol=TOL, atol=TOL, err_msg=f"lse seed {seed}")


@pytest.mark.parametrize("seed", range(12))
def test_random_batch_fp8_matches_the_oracle(seed):
    # kv capped lower than above: the oracle's encoder (a search over the
    # code table for every value) is the slow part of this test
    w, opts, _ = random_batch(seed, cap=400)
    s = w.spec
    ps = s.page_size
    cfg = cfg_of(w)
    o = B.options(prefill_min_rows=-1, kv_chunk=opts.kv_chunk if opts else 0,
                  disable_cascade=opts.disable_cascade if opts else 0,
                  target_ctas=opts.target_ctas if opts else 0)
    gen = torch.Generator().manual_seed(20_000 + seed)
    n_slots = w.num_pages * ps
    k_pool = torch.randn((n_slots, s.n_kv_heads, s.head_dim), generator=gen).to(torch.bfloat16)
    v_pool = torch.randn((n_slots, s.n_kv_heads, s.head_dim), generator=gen).to(torch.bfloat16)
    q = torch.randn((w.total_q, s.n_q_heads, s.head_dim), generator=gen).to(torch.bfloat16)
    kn = torch.randn((w.total_q, s.n_kv_heads, s.head_dim), generator=gen).to(torch.bfloat16)
    vn = torch.randn((w.total_q, s.n_kv_heads, s.head_dim), generator=gen).to(torch.bfloat16)
    pool_slots = np.arange(n_slots, dtype=np.int32)
    new_slots = B.slot_mapping(w.requests, w.block_table, cfg, w.total_q).astype(np.int32)

    shape = (w.num_pages, s.n_kv_heads, ps, s.head_dim)
    ok8, ov8 = np.zeros(shape, np.uint8), np.zeros(shape, np.uint8)
    oks, ovs = np.zeros(shape[:3], np.float32), np.zeros(shape[:3], np.float32)
    F.append_scatter_fp8(ok8, ov8, oks, ovs, k_pool.float().numpy(), v_pool.float().numpy(),
                         pool_slots, ps)
    F.append_scatter_fp8(ok8, ov8, oks, ovs, kn.float().numpy(), vn.float().numpy(),
                         new_slots, ps)
    o_ref, l_ref = OA.mixed_attention(q.float().numpy(), F.dequantize_rows(ok8, oks),
                                      F.dequantize_rows(ov8, ovs), w.requests, w.block_table, ps)

    k8 = torch.full(shape, 0x7F, dtype=torch.uint8, device="cuda")   # e4m3 NaN
    v8 = torch.full(shape, 0x7F, dtype=torch.uint8, device="cuda")
    ks = torch.full(shape[:3], float("nan"), device="cuda")
    vs = torch.full(shape[:3], float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.kv_append_fp8(k8, v8, ks, vs, k_pool.cuda(), v_pool.cuda(),
                    torch.from_numpy(pool_slots).cuda(), cfg, status)
    if w.total_q:
        B.kv_append_fp8(k8, v8, ks, vs, kn.cuda(), vn.cuda(), torch.from_numpy(new_slots).cuda(),
                        cfg, status)
    plan = B.Plan(w.requests, w.block_table, cfg, device="cuda", opts=o)
    assert plan.info.n_prefill_items == 0
    out = torch.full((max(w.total_q, 1), s.n_q_heads, s.head_dim), float("nan"),
                     dtype=torch.bfloat16, device="cuda")
    lse = torch.full((max(w.total_q, 1), s.n_q_heads), float("nan"), device="cuda")
    bt = torch.from_numpy(np.ascontiguousarray(w.block_table)).cuda()
    plan.forward_fp8(q.cuda() if w.total_q else out, k8, v8, ks, vs, bt, out, lse)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert plan.device_status() == 0
    plan.close()

    assert np.array_equal(k8.cpu().numpy(), ok8)
    assert np.array_equal(v8.cpu().numpy(), ov8)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), oks.view(np.uint32))
    assert np.array_equal(vs.cpu().numpy().view(np.uint32), ovs.view(np.uint32))

    rows = np.zeros(max(w.total_q, 1), dtype=bool)
    for qs, qe, _ in w.requests.tolist():
        rows[qs:qe] = True
    if not rows.any():
        return
    got = out.double().cpu().numpy()[rows]
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, o_ref[rows[:w.total_q]], rtol=TOL, atol=TOL,
                               err_msg=f"fp8 seed {seed}")
    np.testing.assert_allclose(lse.double().cpu().numpy()[rows], l_ref[rows[:w.total_q]],
                               rtol=TOL, atol=TOL, err_msg=f"fp8 lse seed {seed}")
