"""Launch order on one stream: kernels that start under the previous one's tail.

The split-KV kernel is launched with programmatic dependent launch. Behind
the KV append it streams history tiles at once, and waits for the append
before it reads q, a tile holding this step's rows, or writes anything.
Behind its own forward's prefill kernel it runs beside it on the SMs the
prefill grid leaves free. The appends start under the previous kernel and
wait for it before they touch memory.

These tests run several layers back to back with nothing between the
launches (one plan, one cache per layer, distinct values per layer; caches
poisoned with NaN before the history is written, so a tile read before its
rows were appended shows up). Every layer is checked against the fp64
oracle. The prefill grid's share of the SMs must not change any bit.
"""

import dataclasses

import numpy as np
import pytest
import torch

from continuous_batching_paged_varlen_gb300 import binding as B
from continuous_batching_paged_varlen_gb300 import workloads as W
from tests.gpu_harness import (assert_request_close, cfg_of, custom_workload, fill_cache,
                               poisoned_cache, run_forward)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from continuous_batching_paged_varlen_gb300 import build
    build.build()
    B.lib()


def layer_values(w, seed):
    """Same requests, pages and prefix sharing as w; new N(0, 1) bf16 values."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)

    def rnd(t):
        return torch.randn(tuple(t.shape), generator=gen, dtype=torch.float32).to(torch.bfloat16)

    q, kn, vn, kh, vh = (rnd(t) for t in (w.q, w.k_new, w.v_new, w.k_hist, w.v_hist))
    sp = w.spec.shared_prefix
    if sp:  # shared positions are one physical copy: the same values for every sharer
        h0 = int(w.hist_requests[0, 0])
        for r in range(1, w.n_requests):
            hs = int(w.hist_requests[r, 0])
            kh[hs:hs + sp] = kh[h0:h0 + sp]
            vh[hs:hs + sp] = vh[h0:h0 + sp]
    return dataclasses.replace(w, q=q, k_new=kn, v_new=vn, k_hist=kh, v_hist=vh)


def _history_caches(layers, cfg):
    caches = []
    for wl in layers:
        kc, vc = poisoned_cache(wl, "cuda")
        n_hist = int(wl.hist_requests[:, 1].max()) if len(wl.hist_requests) else 0
        if n_hist:
            hs = torch.from_numpy(B.slot_mapping(wl.hist_requests, wl.block_table, cfg, n_hist))
            B.kv_append(kc, vc, wl.k_hist.cuda(), wl.v_hist.cuda(), hs.cuda(), cfg)
        caches.append((kc, vc))
    torch.cuda.synchronize()
    return caches


def _check_all(w, out, lse):
    for r in range(w.n_requests):
        m = int(w.requests[r, 1] - w.requests[r, 0])
        if m == 0:
            continue
        if m > 256:
            for rows in ((0, 128), (m - 128, m)):
                assert_request_close(w, out, lse, r, heads=[0, w.spec.n_q_heads - 1], rows=rows)
        else:
            assert_request_close(w, out, lse, r)


def _run_layers(name_or_w, n_layers, rope=False, opts=None):
    w0 = W.make_workload(name_or_w) if isinstance(name_or_w, str) else name_or_w
    layers = [w0] + [layer_values(w0, 1000 + l) for l in range(1, n_layers)]
    cfg = cfg_of(w0)
    caches = _history_caches(layers, cfg)
    s = w0.spec
    slots = torch.from_numpy(B.slot_mapping(w0.requests, w0.block_table, cfg, w0.total_q)).cuda()
    bt = torch.from_numpy(np.ascontiguousarray(w0.block_table)).cuda()
    dev_in = [(wl.q.cuda(), wl.k_new.cuda(), wl.v_new.cuda()) for wl in layers]
    outs = [(torch.full((w0.total_q, s.n_q_heads, s.head_dim), float("nan"), dtype=torch.bfloat16,
                        device="cuda"),
             torch.full((w0.total_q, s.n_q_heads), float("nan"), device="cuda"))
            for _ in layers]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if rope:
        pos = torch.from_numpy(B.positions(w0.requests, w0.total_q)).cuda()
        table = torch.from_numpy(B.rope_table(int(w0.requests[:, 2].max()) + 1, s.head_dim)).cuda()
    plan = B.Plan(w0.requests, w0.block_table, cfg, device="cuda", opts=opts)
    torch.cuda.synchronize()
    # every layer's append and forward back to back: no copy, sync or other
    # launch between them
    for (q, kn, vn), (kc, vc), (o, l) in zip(dev_in, caches, outs):
        if rope:
            B.rope_kv_append(q, kc, vc, kn, vn, pos, slots, table, cfg, status)
        else:
            B.kv_append(kc, vc, kn, vn, slots, cfg, status)
        plan.forward(q, kc, vc, bt, o, l)
    torch.cuda.synchronize()
    assert status.item() == 0 and plan.device_status() == 0
    plan.close()
    return layers, dev_in, outs, caches, slots


@pytest.mark.parametrize("name", ["shared_prefix_decode", "tiny_mixed", "spec_decode_k3"])
def test_layers_back_to_back_match_the_oracle(name):
    layers, _, outs, _, _ = _run_layers(name, 4)
    for wl, (o, l) in zip(layers, outs):
        _check_all(wl, o, l)


def test_rotary_append_then_forward_back_to_back():
    # the rotary append rewrites q in place: the forward behind it must read
    # the rotated rows (it waits for the append before its Q loads)
    from oracle import rope as OR
    w0 = custom_workload([(1, 300), (1, 517), (3, 700), (1, 65)], n_q_heads=8, n_kv_heads=2,
                         head_dim=128, page_size=16, seed=11)
    layers, dev_in, outs, caches, slots = _run_layers(w0, 3, rope=True)
    s = w0.spec
    pos = B.positions(w0.requests, w0.total_q)
    table = B.rope_table(int(w0.requests[:, 2].max()) + 1, s.head_dim).astype(np.float64)
    ps = s.page_size
    sl = slots.long()
    for wl, (q_dev, _, _), (kc, _), (o, l) in zip(layers, dev_in, caches, outs):
        # q_dev now holds the rotated rows: one bf16 unit of the oracle's rotation
        q_ref = OR.rotate(wl.q.double().numpy(), pos, table)
        q_gpu = q_dev.cpu()
        np.testing.assert_allclose(q_gpu.double().numpy(), q_ref, rtol=2.0 ** -7, atol=1e-6)
        # attention over the rotated q and the rotated new k the cache holds
        k_rot = kc[sl // ps, :, sl % ps, :].cpu()
        wr = dataclasses.replace(wl, q=q_gpu, k_new=k_rot)
        _check_all(wr, o, l)


def test_prefill_share_of_the_sms_changes_no_bit():
    # a chunk beside decodes (prefill and split-KV kernels overlapping): the
    # prefill grid's size only moves work items between CTAs
    w = custom_workload([(512, 1536), (1, 900), (1, 1300), (2, 2000), (1, 700)],
                        n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=64, seed=5)
    kc, vc, cfg = fill_cache(w)
    ref = None
    for pc in (0, -1, 1, 3, 7):
        out, lse, st, info = run_forward(w, kc, vc, cfg, B.options(prefill_ctas=pc))
        assert st == 0 and info["n_prefill_items"] > 0 and info["n_decode_items"] > 0
        if pc > 0:
            assert info["prefill_ctas"] == min(pc, info["n_prefill_items"])
        if ref is None:
            ref = (out, lse)
            _check_all(w, out, lse)
        else:
            assert torch.equal(out.view(torch.int16), ref[0].view(torch.int16)), pc
            assert torch.equal(lse.view(torch.int32), ref[1].view(torch.int32)), pc


def test_chunk_beside_decodes_over_layers():
    # prefill + split-KV behind it, then the next layer's append behind the
    # split-KV kernel, which must not complete before the prefill does
    w = custom_workload([(384, 2048), (1, 3000), (1, 1100), (1, 2500)], n_q_heads=8,
                        n_kv_heads=2, head_dim=128, page_size=64, seed=9)
    layers, _, outs, _, _ = _run_layers(w, 3, opts=B.options(prefill_ctas=2))
    for wl, (o, l) in zip(layers, outs):
        _check_all(wl, o, l)
