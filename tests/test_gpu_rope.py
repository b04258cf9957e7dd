"""GPU parity of the fused rotary embedding + KV append (``mb_rope_kv_append``)
against the fp64 oracle (``oracle/rope.py``), through the C ABI.

The kernel computes each rotation in fp32 and rounds once to bf16; the oracle
computes it in fp64 from the same fp32 angle table. One bf16 rounding of a
value differs from its exact value by at most half a unit in the last place,
and the fp32 error before it can move a result across one rounding boundary,
so rotated values must agree to one bf16 unit: |gpu - ref| <= 2^-7 |ref|
(+1e-6 absolute for results that cancel to ~0). V is copied bit for bit and
every slot the call does not own must keep its (NaN) poison.
"""

import numpy as np
import pytest
import torch

from continuous_batching_paged_varlen_gb300 import binding as B
from continuous_batching_paged_varlen_gb300 import workloads as W
from oracle import attention as OA
from oracle import rope as OR
from tests.gpu_harness import BF16_NAN, TOL, cfg_of, custom_workload, poisoned_cache

pytestmark = pytest.mark.gpu

RTOL = 2.0 ** -7
ATOL = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from continuous_batching_paged_varlen_gb300 import build
    build.build()
    B.lib()


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def f64(t):
    return t.to(torch.float64).cpu().numpy()


def run_fused(w, positions, slots, table, q=None, k_new=None, v_new=None):
    s = w.spec
    cfg = cfg_of(w)
    kc, vc = poisoned_cache(w, "cuda")
    q_dev = (w.q if q is None else q).to("cuda").clone()
    kn = (w.k_new if k_new is None else k_new).to("cuda")
    vn = (w.v_new if v_new is None else v_new).to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tab = torch.from_numpy(table).to("cuda")
    B.rope_kv_append(q_dev, kc, vc, kn, vn, torch.from_numpy(positions).to("cuda"),
                     torch.from_numpy(slots).to("cuda"), tab, cfg, status)
    torch.cuda.synchronize()
    return q_dev, kc, vc, int(status.item())


def check_against_oracle(w, positions, slots, table, q_dev, kc, vc, q_in=None, k_in=None,
                         v_in=None):
    s = w.spec
    q_in = w.q if q_in is None else q_in
    k_in = w.k_new if k_in is None else k_in
    v_in = w.v_new if v_in is None else v_in
    shape = (w.num_pages, s.n_kv_heads, s.page_size, s.head_dim)
    kref = np.full(shape, np.nan)
    vref_bits = np.full(shape, BF16_NAN, np.uint16)
    valid = positions >= 0
    qr = OR.rotate(f64(q_in)[valid], positions[valid], table)
    kr = OR.rotate(f64(k_in)[valid], positions[valid], table)
    vin_bits = bits(v_in)
    for j, t in enumerate(np.nonzero(valid)[0].tolist()):
        slot = int(slots[t])
        if slot < 0:
            continue
        page, off = divmod(slot, s.page_size)
        kref[page, :, off] = kr[j]
        vref_bits[page, :, off] = vin_bits[t]
    # Q: rotated rows where the position is valid, untouched elsewhere
    got_q = f64(q_dev)
    np.testing.assert_allclose(got_q[valid], qr, rtol=RTOL, atol=ATOL)
    np.testing.assert_array_equal(bits(q_dev)[~valid], bits(q_in)[~valid])
    # K: rotated at written slots, poison elsewhere
    got_k = f64(kc)
    written = ~np.isnan(kref)
    np.testing.assert_allclose(got_k[written], kref[written], rtol=RTOL, atol=ATOL)
    assert np.all(bits(kc)[~written] == BF16_NAN)
    # V: bit-exact copy, poison elsewhere
    np.testing.assert_array_equal(bits(vc), vref_bits)


@pytest.mark.parametrize("name", ["tiny_mixed", "llama2_7b_orca_iteration",
                                  "decode_heavy_gqa4"])
def test_fused_rope_append_matches_oracle(name):
    w = W.make_workload(name)
    s = w.spec
    cfg = cfg_of(w)
    positions = B.positions(w.requests, w.total_q)
    slots = B.slot_mapping(w.requests, w.block_table, cfg, w.total_q)
    table = B.rope_table(int(w.requests[:, 2].max()) + 1, s.head_dim)
    q_dev, kc, vc, status = run_fused(w, positions, slots, table)
    assert status == 0
    check_against_oracle(w, positions, slots, table, q_dev, kc, vc)


def test_padding_and_bad_indices():
    w = W.make_workload("tiny_mixed")
    s = w.spec
    cfg = cfg_of(w)
    positions = B.positions(w.requests, w.total_q)
    slots = B.slot_mapping(w.requests, w.block_table, cfg, w.total_q)
    table = B.rope_table(256, s.head_dim)
    slots = slots.copy()
    positions = positions.copy()
    slots[3] = -1                                  # padding: Q rotated, no cache write
    positions[7] = 10_000                          # outside the table: token skipped, flagged
    q_dev, kc, vc, status = run_fused(w, positions, slots, table)
    assert status == 1 << B.MB_ERR_DEVICE_INDEX
    pos_ref = positions.copy()
    pos_ref[7] = -1                                # the oracle view: token 7 untouched
    slots_ref = slots.copy()
    slots_ref[7] = -1
    check_against_oracle(w, pos_ref, slots_ref, table, q_dev, kc, vc)
    # a slot past the pool: flagged, its K/V skipped, its Q still rotated
    slots2 = B.slot_mapping(w.requests, w.block_table, cfg, w.total_q).copy()
    slots2[5] = w.num_pages * s.page_size + 3
    positions2 = B.positions(w.requests, w.total_q)
    q_dev, kc, vc, status = run_fused(w, positions2, slots2, table)
    assert status == 1 << B.MB_ERR_DEVICE_INDEX
    slots2_ref = slots2.copy()
    slots2_ref[5] = -1
    check_against_oracle(w, positions2, slots2_ref, table, q_dev, kc, vc)
    # T = 0 enqueues nothing
    empty = torch.zeros(0, dtype=torch.int32, device="cuda")
    B.rope_kv_append(q_dev, kc, vc, kc, vc, empty, empty, torch.from_numpy(table).cuda(), cfg)


@pytest.mark.parametrize("head_dim", [64, 128])
def test_rotated_cache_feeds_attention(head_dim):
    """History and new rows appended through the fused op, then attention:
    matches the oracle's attention of the rotated Q and K."""
    w = custom_workload([(40, 100), (1, 77), (9, 9)], n_q_heads=8, n_kv_heads=2,
                        head_dim=head_dim, page_size=16, seed=3)
    s = w.spec
    cfg = cfg_of(w)
    table = B.rope_table(128, head_dim)
    tab = torch.from_numpy(table).cuda()
    kc, vc = poisoned_cache(w, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # history rows: positions 0..S0-1 of each request (their Q is not used)
    n_hist = int(w.hist_requests[:, 1].max())
    hpos = B.positions(w.hist_requests, n_hist)
    hslots = B.slot_mapping(w.hist_requests, w.block_table, cfg, n_hist)
    dummy_q = torch.zeros((n_hist, s.n_q_heads, head_dim), dtype=torch.bfloat16, device="cuda")
    B.rope_kv_append(dummy_q, kc, vc, w.k_hist.cuda(), w.v_hist.cuda(),
                     torch.from_numpy(hpos).cuda(), torch.from_numpy(hslots).cuda(), tab, cfg,
                     status)
    pos = B.positions(w.requests, w.total_q)
    slots = B.slot_mapping(w.requests, w.block_table, cfg, w.total_q)
    q = w.q.cuda().clone()
    B.rope_kv_append(q, kc, vc, w.k_new.cuda(), w.v_new.cuda(), torch.from_numpy(pos).cuda(),
                     torch.from_numpy(slots).cuda(), tab, cfg, status)
    plan = B.Plan(w.requests, w.block_table, cfg)
    out = torch.empty((w.total_q, s.n_q_heads, head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.total_q, s.n_q_heads), dtype=torch.float32, device="cuda")
    plan.forward(q, kc, vc, torch.from_numpy(w.block_table).cuda(), out, lse)
    torch.cuda.synchronize()
    assert status.item() == 0 and plan.device_status() == 0
    plan.close()
    g = s.n_q_heads // s.n_kv_heads
    for r, (qs, qe, kv) in enumerate(w.requests.tolist()):
        k_log, v_log = w.logical_kv(r)
        k_rot = OR.rotate(f64(k_log), np.arange(kv), table)
        q_rot = OR.rotate(f64(w.q[qs:qe]), pos[qs:qe], table)
        o_ref, l_ref = OA.attend(q_rot, k_rot, f64(v_log), s.scale)
        np.testing.assert_allclose(f64(out[qs:qe]), o_ref, rtol=TOL, atol=TOL)
        np.testing.assert_allclose(f64(lse[qs:qe]), l_ref, rtol=TOL, atol=TOL)
