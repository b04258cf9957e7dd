"""GPU parity of the fp8 (e4m3) KV cache path through the C ABI.

* ``mb_kv_append_fp8`` against ``oracle.fp8`` bit for bit: codes and scales
  (compared as bit patterns), for seeded workloads and for rows with zeros,
  signed zeros, subnormal-range and very large values; padding slots and the
  bad-slot flag.
* ``mb_attn_forward_fp8`` against the fp64 oracle attention over K/V that the
  oracle quantized and dequantized itself (no value from the CUDA path), at
  atol = rtol = 2e-2, for each softmax layout of the kernel (<= 32, <= 64 and
  > 64 query rows per CTA), shared-prefix cascade groups, key ranges split
  into partials, head_dim 64 / 128, page sizes 16 to 128 and GQA 1 to 8.
Caches start as NaN codes and NaN scales, so a read of an unwritten slot
that reaches an output fails.
"""

import math
import zlib

import numpy as np
import pytest
import torch

from continuous_batching_paged_varlen_gb300 import binding as B
from continuous_batching_paged_varlen_gb300 import workloads as W
from oracle import attention as OA
from oracle import fp8 as F
from tests.gpu_harness import TOL, cfg_of, custom_workload

pytestmark = pytest.mark.gpu

SPLIT_KV_ONLY = dict(prefill_min_rows=-1)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from continuous_batching_paged_varlen_gb300 import build
    build.build()
    B.lib()


def slots_of(reqs, block_table, ps):
    """Cache slot of every new row (written out here from the paging rule:
    row i of a request with q rows and kv_length L sits at position
    L - q + i, in page block_table[p // ps], offset p % ps)."""
    total = int(reqs[:, 1].max()) if len(reqs) else 0
    out = np.full(total, -1, np.int64)
    for r, (qs, qe, kv) in enumerate(reqs.tolist()):
        for i in range(qe - qs):
            p = kv - (qe - qs) + i
            out[qs + i] = int(block_table[r][p // ps]) * ps + p % ps
    return out


def empty_caches(w, device="cuda"):
    s = w.spec
    shape = (w.num_pages, s.n_kv_heads, s.page_size, s.head_dim)
    k8 = torch.full(shape, 0x7F, dtype=torch.uint8, device=device)   # e4m3 NaN
    v8 = torch.full(shape, 0x7F, dtype=torch.uint8, device=device)
    ks = torch.full(shape[:3], float("nan"), dtype=torch.float32, device=device)
    vs = torch.full(shape[:3], float("nan"), dtype=torch.float32, device=device)
    return k8, v8, ks, vs


def fill_fp8(w, device="cuda"):
    cfg = cfg_of(w)
    k8, v8, ks, vs = empty_caches(w, device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    ps = w.spec.page_size
    if len(w.k_hist):
        hs = slots_of(w.hist_requests, w.block_table, ps)
        B.kv_append_fp8(k8, v8, ks, vs, w.k_hist.to(device), w.v_hist.to(device),
                        torch.from_numpy(hs.astype(np.int32)).to(device), cfg, status)
    ns = slots_of(w.requests, w.block_table, ps)
    B.kv_append_fp8(k8, v8, ks, vs, w.k_new.to(device), w.v_new.to(device),
                    torch.from_numpy(ns.astype(np.int32)).to(device), cfg, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return k8, v8, ks, vs, cfg


def oracle_caches(w):
    s = w.spec
    shape = (w.num_pages, s.n_kv_heads, s.page_size, s.head_dim)
    k8 = np.full(shape, 0x7F, np.uint8)
    v8 = np.full(shape, 0x7F, np.uint8)
    ks = np.full(shape[:3], np.nan, np.float32)
    vs = np.full(shape[:3], np.nan, np.float32)
    f32 = lambda t: t.float().cpu().numpy()  # noqa: E731  (bf16 values, exact in fp32)
    ps = s.page_size
    if len(w.k_hist):
        F.append_scatter_fp8(k8, v8, ks, vs, f32(w.k_hist), f32(w.v_hist),
                             slots_of(w.hist_requests, w.block_table, ps), ps)
    F.append_scatter_fp8(k8, v8, ks, vs, f32(w.k_new), f32(w.v_new),
                         slots_of(w.requests, w.block_table, ps), ps)
    return k8, v8, ks, vs


def bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


# ------------------------------------------------------------------ append

@pytest.mark.parametrize("name", ["tiny_mixed", "shared_prefix_decode",
                                  "llama2_7b_orca_iteration"])
def test_fp8_append_bit_exact(name):
    w = W.make_workload(name)
    k8, v8, ks, vs, _ = fill_fp8(w)
    ok8, ov8, oks, ovs = oracle_caches(w)
    assert np.array_equal(k8.cpu().numpy(), ok8)
    assert np.array_equal(v8.cpu().numpy(), ov8)
    assert np.array_equal(bits(ks.cpu().numpy()), bits(oks))
    assert np.array_equal(bits(vs.cpu().numpy()), bits(ovs))


@pytest.mark.parametrize("head_dim", [64, 128])
def test_fp8_append_special_rows(head_dim):
    hkv, ps, pages = 2, 16, 4
    cfg = B.config(4, hkv, head_dim, ps, pages, 4)
    g = torch.Generator().manual_seed(head_dim)
    T = 12
    x = torch.randn((2, T, hkv, head_dim), generator=g)
    x[0, 0] = 0.0                                              # all-zero rows
    x[0, 1, 0] = -0.0                                          # signed zeros
    x[0, 1, 0, 3] = 1.0
    x[0, 2] *= 1e-30                                           # tiny magnitudes
    x[0, 3] *= 1e30                                            # huge magnitudes
    x[0, 4, 1, :] = torch.tensor([3.3895e38] + [1e-38] * (head_dim - 1))  # near bf16 max
    x[0, 5] = torch.where(torch.rand(x[0, 5].shape, generator=g) < 0.9, 0.0, x[0, 5])
    x[1, 6] = -x[1, 6].abs()                                  # one sign only
    xb = x.to(torch.bfloat16)
    kn, vn = xb[0], xb[1]
    slots = np.array([0, 5, 17, 18, 33, 63, 40, 41, 42, 43, 44, 45], np.int64)
    k8 = torch.full((pages, hkv, ps, head_dim), 0xAB, dtype=torch.uint8, device="cuda")
    v8 = k8.clone()
    ks = torch.full((pages, hkv, ps), -7.0, dtype=torch.float32, device="cuda")
    vs = ks.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.kv_append_fp8(k8, v8, ks, vs, kn.cuda(), vn.cuda(),
                    torch.from_numpy(slots.astype(np.int32)).cuda(), cfg, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    ok8 = np.full((pages, hkv, ps, head_dim), 0xAB, np.uint8)
    ov8 = ok8.copy()
    oks = np.full((pages, hkv, ps), -7.0, np.float32)
    ovs = oks.copy()
    F.append_scatter_fp8(ok8, ov8, oks, ovs, kn.float().numpy(), vn.float().numpy(), slots, ps)
    assert np.array_equal(k8.cpu().numpy(), ok8)
    assert np.array_equal(v8.cpu().numpy(), ov8)
    assert np.array_equal(bits(ks.cpu().numpy()), bits(oks))
    assert np.array_equal(bits(vs.cpu().numpy()), bits(ovs))


def test_fp8_append_padding_and_bad_slot_flag():
    hkv, d, ps, pages = 2, 64, 16, 3
    cfg = B.config(2, hkv, d, ps, pages, 3)
    kn = torch.randn(3, hkv, d, device="cuda").to(torch.bfloat16)
    vn = torch.randn(3, hkv, d, device="cuda").to(torch.bfloat16)
    k8 = torch.zeros((pages, hkv, ps, d), dtype=torch.uint8, device="cuda")
    v8 = torch.zeros_like(k8)
    ks = torch.zeros((pages, hkv, ps), dtype=torch.float32, device="cuda")
    vs = torch.zeros_like(ks)
    slots = torch.tensor([7, -1, pages * ps + 1], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.kv_append_fp8(k8, v8, ks, vs, kn, vn, slots, cfg, status)
    torch.cuda.synchronize()
    assert status.item() == 1 << B.MB_ERR_DEVICE_INDEX
    c, s = F.quantize_rows(kn[0].float().cpu().numpy())
    assert np.array_equal(k8[0, :, 7].cpu().numpy(), c)
    assert np.array_equal(bits(ks[0, :, 7].cpu().numpy()), bits(s))
    assert int((ks != 0).sum()) == hkv and int((vs != 0).sum()) == hkv
    # T = 0 enqueues nothing
    B.kv_append_fp8(k8, v8, ks, vs, kn, vn, slots[:0], cfg, status)


# --------------------------------------------------------------- attention

def oracle_fp8_request(w, r):
    """fp64 attention of request r over its K/V as the oracle quantizes and
    dequantizes them."""
    qs, qe, kv = [int(x) for x in w.requests[r]]
    k, v = w.logical_kv(r)
    kd = F.dequantize_rows(*F.quantize_rows(k.float().cpu().numpy()))
    vd = F.dequantize_rows(*F.quantize_rows(v.float().cpu().numpy()))
    q = w.q[qs:qe].to(torch.float64).cpu().numpy()
    s = w.spec
    g = s.n_q_heads // s.n_kv_heads
    outs, lses = [], []
    for h in range(s.n_q_heads):
        o, l = OA.attend(q[:, h:h + 1], kd[:, h // g:h // g + 1], vd[:, h // g:h // g + 1],
                         s.scale)
        outs.append(o[:, 0])
        lses.append(l[:, 0])
    return np.stack(outs, 1), np.stack(lses, 1)


def run_fp8(w, opts=SPLIT_KV_ONLY):
    k8, v8, ks, vs, cfg = fill_fp8(w)
    plan = B.Plan(w.requests, w.block_table, cfg, opts=B.options(**opts))
    s = w.spec
    out = torch.full((w.total_q, s.n_q_heads, s.head_dim), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    lse = torch.full((w.total_q, s.n_q_heads), float("nan"), dtype=torch.float32, device="cuda")
    bt = torch.from_numpy(np.ascontiguousarray(w.block_table)).cuda()
    plan.forward_fp8(w.q.cuda(), k8, v8, ks, vs, bt, out, lse)
    torch.cuda.synchronize()
    status = plan.device_status()
    info = plan.info.as_dict()
    plan.close()
    return out, lse, status, info


def check_all(w, out, lse):
    o = out.to(torch.float64).cpu().numpy()
    ls = lse.to(torch.float64).cpu().numpy()
    for r in range(w.n_requests):
        qs, qe, _ = [int(x) for x in w.requests[r]]
        if qe == qs:
            continue
        o_ref, l_ref = oracle_fp8_request(w, r)
        assert np.isfinite(o[qs:qe]).all(), f"non-finite output in request {r}"
        np.testing.assert_allclose(o[qs:qe], o_ref, rtol=TOL, atol=TOL, err_msg=f"request {r}")
        np.testing.assert_allclose(ls[qs:qe], l_ref, rtol=TOL, atol=TOL,
                                   err_msg=f"lse request {r}")


def _draw(rng, n, q, lo, hi):
    return [(q, int(rng.integers(max(lo, q), hi + 1))) for _ in range(n)]


rng = np.random.default_rng(8)
CASES = {
    # (shapes, Hq, Hkv, D, ps, shared_prefix)
    "decode_gqa4_d128": (_draw(rng, 12, 1, 1, 3000), 16, 4, 128, 64, 0),     # 4 rows / CTA
    "decode_gqa1_d64": (_draw(rng, 9, 1, 1, 700), 4, 4, 64, 16, 0),          # 1 row / CTA
    "spec_decode_gqa8": (_draw(rng, 6, 4, 4, 1500), 16, 2, 128, 32, 0),      # 32 rows / CTA
    "rows_48_per_cta": (_draw(rng, 5, 12, 12, 900), 8, 2, 64, 128, 0),       # 2 copies
    "rows_96_per_cta": (_draw(rng, 4, 24, 24, 800), 8, 2, 128, 64, 0),       # 1 copy, 2 passes
    "rows_160_split": ([(40, 300), (40, 1000)], 8, 2, 64, 16, 0),            # 128 + 32 rows
    "long_keys_partials": ([(1, 20000), (2, 9000), (1, 130)], 8, 2, 128, 64, 0),
    "shared_prefix": ([(1, 300 + 17 * i) for i in range(10)], 8, 2, 128, 16, 256),
    "shared_prefix_many": ([(2, 200 + 3 * i) for i in range(20)], 16, 4, 64, 32, 128),
}
# CTAs of at most 8 rows with head_dim 128 run the few-row form of the
# kernel (keys as the MMA's M, rows as its N), built for 4 and 8 rows
rng_t = np.random.default_rng(81)
FEW_ROW_CASES = {
    # (shapes, Hq, Hkv, D, ps, shared_prefix, build rows)
    "few_rows_4_ps128": (_draw(rng_t, 7, 1, 1, 6000), 8, 2, 128, 128, 0, 4),
    "few_rows_8_ps32": (_draw(rng_t, 10, 1, 1, 5000), 16, 2, 128, 32, 0, 8),
    "few_rows_8_spec_ps16": (_draw(rng_t, 8, 4, 4, 2500), 8, 4, 128, 16, 0, 8),
    "few_rows_8_cascade": ([(1, 400 + 13 * i) for i in range(4)], 4, 2, 128, 128, 256, 8),
    "few_rows_3_of_4_split": ([(1, 30000), (1, 129), (1, 128), (1, 1)], 12, 4, 128, 64, 0, 4),
}
CASES.update({k: v[:6] for k, v in FEW_ROW_CASES.items()})
# the same batch shapes with more rows per CTA run the form with rows in TMEM lanes
CASES.update({
    "spec_16_rows_ps16": (_draw(rng_t, 8, 4, 4, 2500), 16, 4, 128, 16, 0),
    "cascade_24_rows_ps128": ([(1, 400 + 13 * i) for i in range(6)], 8, 2, 128, 128, 256),
})


@pytest.mark.parametrize("case", sorted(CASES))
def test_fp8_attention_matches_oracle(case):
    shapes, hq, hkv, d, ps, shared = CASES[case]
    w = custom_workload(shapes, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, page_size=ps,
                        seed=zlib.crc32(case.encode()) % 1000, shared_prefix=shared)
    out, lse, status, info = run_fp8(w)
    assert status == 0
    assert info["n_prefill_items"] == 0
    if shared:
        assert info["n_cascade_groups"] >= 1
    check_all(w, out, lse)


@pytest.mark.parametrize("case", sorted(FEW_ROW_CASES))
def test_fp8_few_row_build_chosen(case):
    shapes, hq, hkv, d, ps, shared, rows = FEW_ROW_CASES[case]
    w = custom_workload(shapes, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, page_size=ps,
                        seed=zlib.crc32(case.encode()) % 1000, shared_prefix=shared)
    out, lse, status, info = run_fp8(w)
    assert status == 0
    # the largest CTA sets the build (4, 8, 16 or 32 rows)
    assert rows // 2 < info["splitkv_max_rows"] <= rows
    check_all(w, out, lse)


FP8_PREFILL_CASES = {
    # (shapes, Hq, Hkv, D, ps, shared_prefix): prefill requests on the
    # tensor-core kernel over bf16 staging pages, decodes beside them
    "tiny_mixed_shape": ([(96, 96), (1, 200), (32, 160)], 4, 2, 64, 16, 0),
    "chunk_and_decodes_d128": ([(300, 1900), (1, 700), (1, 1500), (2, 2300)], 8, 2, 128, 64, 0),
    "prefills_sharing_pages": ([(64, 320), (48, 304), (40, 296)], 8, 4, 128, 16, 256),
}


@pytest.mark.parametrize("case", sorted(FP8_PREFILL_CASES))
def test_fp8_prefill_on_tensor_cores_matches_oracle(case):
    shapes, hq, hkv, d, ps, shared = FP8_PREFILL_CASES[case]
    w = custom_workload(shapes, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, page_size=ps,
                        seed=zlib.crc32(case.encode()) % 1000, shared_prefix=shared)
    out, lse, status, info = run_fp8(w, opts=dict(fp8_cache=1))
    assert status == 0
    assert info["n_prefill_items"] > 0 and info["staged_pages"] > 0
    # every page the prefill requests map is staged once
    m = w.requests[:, 1] - w.requests[:, 0]
    pre = np.nonzero(m >= 16)[0]
    pages = {int(w.block_table[r][b]) for r in pre
             for b in range(-(-int(w.requests[r, 2]) // ps))}
    assert info["staged_pages"] == len(pages)
    check_all(w, out, lse)


@pytest.mark.parametrize("name", ["decode_heavy_gqa4", "spec_decode_k3", "shared_prefix_decode"])
def test_fp8_decode_batches_sampled(name):
    # the full decode batches the bench times on the fp8 cache (the planner's
    # own options), sampled requests against the oracle over its dequantized
    # K/V
    w = W.make_workload(name, device="cuda")
    out, lse, status, info = run_fp8(w, opts=dict(fp8_cache=1))
    assert status == 0 and info["n_prefill_items"] == 0
    o = out.to(torch.float64).cpu().numpy()
    ls = lse.to(torch.float64).cpu().numpy()
    assert np.isfinite(o).all()
    rng = np.random.default_rng(5)
    k = min(10, w.n_requests)
    for r in sorted(set(rng.choice(w.n_requests, k, replace=False).tolist()) | {0, w.n_requests - 1}):
        qs, qe, _ = [int(x) for x in w.requests[r]]
        o_ref, l_ref = oracle_fp8_request(w, r)
        np.testing.assert_allclose(o[qs:qe], o_ref, rtol=TOL, atol=TOL, err_msg=f"request {r}")
        np.testing.assert_allclose(ls[qs:qe], l_ref, rtol=TOL, atol=TOL,
                                   err_msg=f"lse request {r}")


@pytest.mark.parametrize("name,reqs", [("chunked_prefill_mix", (0, 1, 40, 64)),
                                       ("llama2_7b_orca_iteration", (0, 1, 2)),
                                       ("varlen_prefill", (0, 5, 11, 15))])
def test_fp8_prefill_batches_sampled(name, reqs):
    # the full chunk (2048 rows at kv 32768) or prompt (4096 rows) on the
    # tensor-core kernel over staged pages and the decodes beside it; sampled
    # heads / rows against the oracle
    w = W.make_workload(name)
    out, lse, status, info = run_fp8(w, opts=dict(fp8_cache=1))
    assert status == 0 and info["n_prefill_items"] > 0 and info["staged_pages"] > 0
    s = w.spec
    g = s.n_q_heads // s.n_kv_heads
    o = out.to(torch.float64).cpu().numpy()
    ls = lse.to(torch.float64).cpu().numpy()
    for r in reqs:
        qs, qe, kv = [int(x) for x in w.requests[r]]
        k, v = w.logical_kv(r)
        kd = F.dequantize_rows(*F.quantize_rows(k.float().cpu().numpy()))
        vd = F.dequantize_rows(*F.quantize_rows(v.float().cpu().numpy()))
        m = qe - qs
        rows = [(0, min(m, 64)), (max(0, m - 64), m)] if m > 64 else [(0, m)]
        for a, b in rows:
            q = w.q[qs + a:qs + b].to(torch.float64).cpu().numpy()
            for h in (0, 13, s.n_q_heads - 1):
                kh = h // g
                o_ref, l_ref = _attend_rows(q[:, h], kd[:, kh], vd[:, kh], kv - m + a, s.scale)
                np.testing.assert_allclose(o[qs + a:qs + b, h], o_ref, rtol=TOL, atol=TOL,
                                           err_msg=f"request {r} head {h} rows {a}:{b}")
                np.testing.assert_allclose(ls[qs + a:qs + b, h], l_ref, rtol=TOL, atol=TOL)


def test_fp8_a_thousand_short_requests():
    # 1000 short requests of every kind on the fp8 cache (decode work on the
    # codes, the chunks' pages staged for the tensor-core kernel)
    rng = np.random.default_rng(34)
    shapes = [(1, 1)] + [((1, 4, 24)[i % 3], 0) for i in range(999)]
    shapes = [(m, kv if kv else int(rng.integers(m, 301))) for m, kv in shapes]
    w = custom_workload(shapes, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=16, seed=34)
    out, lse, status, info = run_fp8(w, opts=dict(fp8_cache=1))
    assert status == 0 and info["staged_pages"] > 0
    check_all(w, out, lse)


def test_fp8_long_context_sampled():
    # the bf16 long-context case on the fp8 cache: a 131072-key decode (128
    # partials per row with a 1024-key chunk), a 65537-key decode and a
    # 300-row chunk over a 100k-key history, whose pages are staged for the
    # tensor-core kernel
    w = custom_workload([(1, 131072), (300, 100000), (1, 65537)], n_q_heads=8, n_kv_heads=2,
                        head_dim=128, page_size=64, seed=21)
    s = w.spec
    g = s.n_q_heads // s.n_kv_heads
    for opts in (dict(fp8_cache=1), dict(fp8_cache=1, kv_chunk=1024)):
        out, lse, status, info = run_fp8(w, opts=opts)
        assert status == 0 and info["staged_pages"] > 0
        o = out.to(torch.float64).cpu().numpy()
        ls = lse.to(torch.float64).cpu().numpy()
        for r, rows, heads in ((0, [(0, 1)], range(8)), (2, [(0, 1)], range(8)),
                               (1, [(0, 16), (284, 300)], (0, 5))):
            qs, qe, kv = [int(x) for x in w.requests[r]]
            k, v = w.logical_kv(r)
            kd = F.dequantize_rows(*F.quantize_rows(k.float().cpu().numpy()))
            vd = F.dequantize_rows(*F.quantize_rows(v.float().cpu().numpy()))
            m = qe - qs
            for a, b in rows:
                q = w.q[qs + a:qs + b].to(torch.float64).cpu().numpy()
                for h in heads:
                    o_ref, l_ref = _attend_rows(q[:, h], kd[:, h // g], vd[:, h // g], kv - m + a,
                                                s.scale)
                    np.testing.assert_allclose(o[qs + a:qs + b, h], o_ref, rtol=TOL, atol=TOL,
                                               err_msg=f"request {r} head {h} rows {a}:{b}")
                    np.testing.assert_allclose(ls[qs + a:qs + b, h], l_ref, rtol=TOL, atol=TOL)


def _attend_rows(q, k, v, first_pos, scale):
    """fp64 attention of query rows q [n, D] at positions first_pos..first_pos
    + n - 1 over keys k, v [>= first_pos + n, D] (row i sees keys <= its
    position), through the oracle's own routine: the rows are the last n new
    rows of a request whose history is everything before first_pos."""
    n = q.shape[0]
    kv = first_pos + n
    o, l = OA.attend(q[:, None, :], k[:kv, None, :], v[:kv, None, :], scale)
    return o[:, 0], l[:, 0]


def test_fp8_forward_rejects_prefill_plans():
    w = custom_workload([(200, 200), (1, 50)], n_q_heads=4, n_kv_heads=2, head_dim=64,
                        page_size=16)
    k8, v8, ks, vs, cfg = fill_fp8(w)
    plan = B.Plan(w.requests, w.block_table, cfg)
    assert plan.info.n_prefill_items > 0
    out = torch.empty((w.total_q, 4, 64), dtype=torch.bfloat16, device="cuda")
    bt = torch.from_numpy(np.ascontiguousarray(w.block_table)).cuda()
    with pytest.raises(B.MBError):
        plan.forward_fp8(w.q.cuda(), k8, v8, ks, vs, bt, out, None)
    plan.close()


def test_fp8_matches_bf16_path_closely():
    """The fp8 forward and the bf16 forward over the dequantized cache agree
    (same arithmetic up to the f16 rounding of q)."""
    w = custom_workload(_draw(np.random.default_rng(3), 8, 1, 1, 2000), n_q_heads=8,
                        n_kv_heads=2, head_dim=128, page_size=32, seed=11)
    out8, lse8, st, _ = run_fp8(w)
    assert st == 0
    # dequantize the oracle-written cache into a bf16 cache and run the bf16 path on it
    ok8, ov8, oks, ovs = oracle_caches(w)
    kd = torch.from_numpy(np.nan_to_num(F.dequantize_rows(ok8, oks))).to(torch.bfloat16).cuda()
    vd = torch.from_numpy(np.nan_to_num(F.dequantize_rows(ov8, ovs))).to(torch.bfloat16).cuda()
    plan = B.Plan(w.requests, w.block_table, cfg_of(w), opts=B.options(**SPLIT_KV_ONLY))
    out = torch.empty_like(out8)
    bt = torch.from_numpy(np.ascontiguousarray(w.block_table)).cuda()
    plan.forward(w.q.cuda(), kd, vd, bt, out, None)
    torch.cuda.synchronize()
    plan.close()
    # bf16 rounding of the dequantized values is the only extra error here
    np.testing.assert_allclose(out8.float().cpu().numpy(), out.float().cpu().numpy(),
                               rtol=TOL, atol=TOL)
    assert math.isfinite(float(lse8.sum()))


def test_fp8_split_rows_merged_on_every_forward():
    """The fused merge's arrival counters return to zero after each forward:
    one plan run three times gives the same complete rows."""
    shapes, hq, hkv, d, ps, shared = CASES["shared_prefix"]
    w = custom_workload(shapes, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, page_size=ps,
                        seed=31, shared_prefix=shared)
    k8, v8, ks, vs, cfg = fill_fp8(w)
    plan = B.Plan(w.requests, w.block_table, cfg, opts=B.options(**SPLIT_KV_ONLY, kv_chunk=64))
    assert plan.info.n_combine > 0
    bt = torch.from_numpy(np.ascontiguousarray(w.block_table)).cuda()
    q = w.q.cuda()
    res = []
    for _ in range(3):
        out = torch.full((w.total_q, hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((w.total_q, hq), float("nan"), dtype=torch.float32, device="cuda")
        plan.forward_fp8(q, k8, v8, ks, vs, bt, out, lse)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        res.append((out, lse))
    plan.close()
    for out, lse in res[1:]:
        assert torch.equal(out.view(torch.int16), res[0][0].view(torch.int16))
        assert torch.equal(lse.view(torch.int32), res[0][1].view(torch.int32))
    check_all(w, *res[0])
