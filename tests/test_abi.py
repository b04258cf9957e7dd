"""C ABI and host planner tests (no GPU: only host-side entry points run).

* the library loads and exports every function ``include/mb.h`` declares;
* argument validation returns the documented status codes;
* ``mb_slot_mapping`` places rows where the oracle's addressing does;
* the planner's work lists cover every visible (row, head, key) exactly once,
  send each row's partials to one combine entry, and group shared prefixes.
"""

import ctypes
import math
import os
import re

import numpy as np
import pytest

from continuous_batching_paged_varlen_gb300 import binding as B
from continuous_batching_paged_varlen_gb300 import build as build_mod
from continuous_batching_paged_varlen_gb300 import workloads as W
from oracle import attention as OA
from tests.conftest import ROOT, read_int_table

HEADER = os.path.join(ROOT, "include", "mb.h")
MB_ERR_INVALID_ARG, MB_ERR_SHAPE = 1, 2


@pytest.fixture(scope="module")
def L():
    build_mod.build()
    return B.lib()


def declared_functions():
    inc = os.path.join(ROOT, "include")
    text = "\n".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc))
                     if f.endswith(".h"))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mb_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert {"mb_kv_append", "mb_attn_plan", "mb_attn_forward", "mb_attn_destroy"} <= set(names)
    for n in names:
        assert hasattr(L, n), n
    assert L.mb_abi_version() == 3
    assert L.mb_status_string(0) == b"ok"


def cfg_for(w):
    s = w.spec
    return B.config(s.n_q_heads, s.n_kv_heads, s.head_dim, s.page_size, w.num_pages,
                    w.block_table.shape[1], s.scale or 0.0)


def test_slot_mapping_hand_worked_fixture(L):
    """tests/golden/append_tiny_ps16.txt, worked by hand from the addressing rule."""
    rows = read_int_table("append_tiny_ps16.txt")
    cfg = B.config(1, 1, 64, 16, 8, 3)
    bt = np.array([[5, 2, -1], [0, 7, 4]], dtype=np.int32)
    slots = B.slot_mapping([(0, 3, 18), (3, 4, 33)], bt, cfg, 4)
    assert slots.tolist() == [flat for _, _, _, flat in rows]
    for t, page, slot, flat in rows:
        assert flat == page * 16 + slot


@pytest.mark.parametrize("name", ["tiny_mixed", "llama2_7b_orca_iteration", "decode_heavy_gqa4",
                                  "shared_prefix_decode"])
def test_slot_mapping_matches_oracle_addressing(L, name):
    w = W.make_workload(name, with_values=False)
    cfg = cfg_for(w)
    slots = B.slot_mapping(w.requests, w.block_table, cfg, w.total_q)
    ps = w.spec.page_size
    for r, (qs, qe, kv) in enumerate(w.requests.tolist()):
        s0 = kv - (qe - qs)
        for t in range(qs, qe):
            page, slot = OA.logical_position_location(w.block_table[r], s0 + t - qs, ps)
            assert slots[t] == page * ps + slot
    assert len(set(slots.tolist())) == len(slots)  # no two new rows share a slot


def _plan_status(reqs, bt, cfg, opts=None):
    try:
        B.HostPlan(reqs, bt, cfg, opts)
        return 0
    except B.MBError as e:
        return e.status


def test_validation_errors(L):
    bt = np.array([[0, 1], [2, 3]], dtype=np.int32)
    good = B.config(4, 2, 64, 16, 4, 2)
    ok = [(0, 2, 20), (2, 3, 17)]
    assert _plan_status(ok, bt, good) == 0
    assert _plan_status([(0, 2, 1), (2, 3, 17)], bt, good) == 2        # q_rows > kv_length
    assert _plan_status([(0, 2, 20), (1, 3, 17)], bt, good) == 2       # overlapping q ranges
    assert _plan_status([(0, 2, 40), (2, 3, 17)], bt, good) == 2       # more blocks than columns
    bad_bt = bt.copy()
    bad_bt[1, 1] = 4
    assert _plan_status(ok, bad_bt, good) == 2                         # page id out of the pool
    assert _plan_status([(3, 2, 20)], bt[:1], good) == 2               # q_end < q_start
    assert _plan_status(ok, bt, B.config(4, 3, 64, 16, 4, 2)) == 2     # Hq % Hkv
    assert _plan_status(ok, bt, B.config(4, 2, 96, 16, 4, 2)) == 3     # head_dim
    assert _plan_status(ok, bt, B.config(4, 2, 64, 24, 4, 2)) == 3     # page size
    assert _plan_status(ok, bt, good, B.options(kv_chunk=100)) == 1    # chunk not /64
    # q_rows = 0 requests are accepted and ignored (their table entries unused)
    assert _plan_status([(0, 0, 0), (0, 1, 17)], np.array([[-1, -1], [2, 3]], np.int32), good) == 0
    # empty batch
    hp = B.HostPlan(np.zeros((0, 3), np.int32), np.zeros((0, 2), np.int32), good)
    assert hp.info.total_q == 0 and hp.info.n_launches == 0
    # slot mapping rejects a total_q smaller than the rows
    with pytest.raises(B.MBError):
        B.slot_mapping(ok, bt, good, 2)


DECODE_ITEM = np.dtype([("bt_row", "<i4"), ("kv_head", "<i4"), ("k_begin", "<i4"),
                        ("k_end", "<i4"), ("row_begin", "<i4"), ("n_rows", "<i4"),
                        ("pad0", "<i4"), ("pad1", "<i4")])
ROW = np.dtype([("q_index", "<i4"), ("q_head", "<i4"), ("vis_end", "<i4"), ("dst", "<i4")])
PREFILL_ITEM = np.dtype([("req", "<i4"), ("q_head", "<i4"), ("q_row0", "<i4"),
                         ("n_rows", "<i4"), ("s0", "<i4"), ("i0", "<i4"),
                         ("kv_length", "<i4"), ("n_kv_tiles", "<i4")])
COMBINE = np.dtype([("q_index", "<i4"), ("q_head", "<i4"), ("slot_begin", "<i4"),
                    ("n_slots", "<i4")])


def decode_plan(hp):
    inf = hp.info
    meta = np.frombuffer(hp.metadata(), dtype=np.uint8)
    off = hp.layout()

    def arr(o, dt, n):
        return np.frombuffer(meta[o:o + n * dt.itemsize].tobytes(), dtype=dt)

    assert np.all(meta[:4] == 0)  # status word starts cleared
    return (arr(off[0], DECODE_ITEM, inf.n_decode_items), arr(off[1], ROW, inf.n_decode_rows),
            arr(off[2], PREFILL_ITEM, inf.n_prefill_items), arr(off[3], COMBINE, inf.n_combine))


def check_coverage(w, opts=None):
    cfg = cfg_for(w)
    hp = B.HostPlan(w.requests, w.block_table, cfg, opts)
    items, rows, pitems, comb = decode_plan(hp)
    inf = hp.info
    s = w.spec
    g = s.n_q_heads // s.n_kv_heads
    ps = s.page_size
    # the largest split-KV CTA, which picks the fp8 kernel's form
    assert inf.splitkv_max_rows == (int(items["n_rows"].max()) if len(items) else 0)
    covered = {}     # (q_index, q_head) -> list of (k_begin, k_end, slot)
    for it in items:
        assert 1 <= it["n_rows"] <= 128
        assert 0 <= it["k_begin"] < it["k_end"]
        for rw in rows[it["row_begin"]:it["row_begin"] + it["n_rows"]]:
            assert rw["q_head"] // g == it["kv_head"]          # one KV head per CTA
            covered.setdefault((int(rw["q_index"]), int(rw["q_head"])), []).append(
                (int(it["k_begin"]), int(it["k_end"]), int(rw["dst"]), int(rw["vis_end"]),
                 int(it["bt_row"])))
    pcover = {}
    for p in pitems:
        assert 1 <= p["n_rows"] <= 256
        for i in range(p["n_rows"]):
            key = (int(p["q_row0"]) + i, int(p["q_head"]))
            assert key not in pcover
            pcover[key] = p
    slot_writes = {}
    comb_by_row = {(int(c["q_index"]), int(c["q_head"])): c for c in comb}
    assert len(comb_by_row) == len(comb)
    for r, (qs, qe, kv) in enumerate(w.requests.tolist()):
        m = qe - qs
        s0 = kv - m
        for i in range(m):
            for h in range(s.n_q_heads):
                key = (qs + i, h)
                if key in pcover:
                    p = pcover[key]
                    assert key not in covered
                    assert p["s0"] == s0 and p["kv_length"] == kv and p["i0"] + (qs + i - p["q_row0"]) == i
                    last = min(kv, s0 + p["i0"] + p["n_rows"])
                    assert p["n_kv_tiles"] == math.ceil(last / 128)
                    # every visible key of the row lies in a visited tile
                    assert p["n_kv_tiles"] * 128 >= s0 + i + 1
                    continue
                segs = sorted(covered[key])
                # the key ranges tile [0, kv) exactly once
                assert segs[0][0] == 0 and segs[-1][1] == kv
                for a, b in zip(segs, segs[1:]):
                    assert a[1] == b[0]
                for kb, ke, dst, vis, btr in segs:
                    assert vis == s0 + i + 1
                    # the addressing row is this request's or shares its pages there
                    nb0, nb1 = kb // ps, (ke - 1) // ps
                    assert np.array_equal(w.block_table[btr, nb0:nb1 + 1],
                                          w.block_table[r, nb0:nb1 + 1])
                if len(segs) == 1:
                    assert segs[0][2] < 0 and key not in comb_by_row
                else:
                    c = comb_by_row[key]
                    assert c["n_slots"] == len(segs)
                    assert sorted(sg[2] for sg in segs) == list(
                        range(c["slot_begin"], c["slot_begin"] + c["n_slots"]))
                    for sg in segs:
                        assert sg[2] not in slot_writes
                        slot_writes[sg[2]] = key
    assert len(slot_writes) == inf.n_partials
    return hp, inf


@pytest.mark.parametrize("name", W.ORDER)
def test_planner_coverage_default(L, name):
    w = W.make_workload(name, with_values=False)
    hp, inf = check_coverage(w)
    if name == "shared_prefix_decode":
        assert inf.n_cascade_groups == 1 and inf.cascade_keys == 4096
    else:
        assert inf.n_cascade_groups == 0
    if name in ("llama2_7b_orca_iteration", "chunked_prefill_mix", "tiny_mixed"):
        assert inf.n_prefill_items > 0


@pytest.mark.parametrize("name", ["tiny_mixed", "shared_prefix_decode", "llama2_7b_orca_iteration"])
@pytest.mark.parametrize("opts", [dict(prefill_min_rows=-1), dict(kv_chunk=64),
                                  dict(kv_chunk=128, disable_cascade=1),
                                  dict(prefill_min_rows=1, kv_chunk=256)])
def test_planner_coverage_options(L, name, opts):
    w = W.make_workload(name, with_values=False)
    check_coverage(w, B.options(**opts))


def test_small_decode_batch_beside_prefill_gets_sms_and_whole_ranges(L):
    # two MHA decodes beside a 4096-row prompt: their 64 (request, head) CTAs
    # are latency-bound, so the planner leaves them SMs next to the prefill
    # grid and keeps each key range whole (one CTA per request and KV head)
    # rather than splitting the ranges into one wave of short CTAs after it
    w = W.make_workload("llama2_7b_orca_iteration", with_values=False)
    inf = B.HostPlan(w.requests, w.block_table, cfg_for(w)).info
    assert inf.n_prefill_items == 512 and 0 < inf.prefill_ctas < 152
    assert inf.n_decode_items == 2 * 32 and inf.n_combine == 0 and inf.n_partials == 0
    assert inf.kv_chunk >= 1700
    # every SM to the prefill grid (the caller's choice): one wave of split
    # CTAs that run in its tail
    inf = B.HostPlan(w.requests, w.block_table, cfg_for(w), B.options(prefill_ctas=-1)).info
    assert inf.prefill_ctas == 152 and inf.n_decode_items > 64 and inf.n_combine == 2 * 32
    # a chunk fixed by the caller is kept
    inf = B.HostPlan(w.requests, w.block_table, cfg_for(w), B.options(kv_chunk=512)).info
    assert inf.kv_chunk == 512


def _host_info(shapes, opts, **kw):
    spec = W.WorkloadSpec(name="custom", requests=tuple(shapes), seed=0, **kw)
    blocks = sum(math.ceil(kv / kw["page_size"]) for _, kv in shapes)
    w = W.make_workload(W.WorkloadSpec(**{**spec.__dict__, "pool_pages": blocks + 3}),
                        with_values=False)
    hp = B.HostPlan(w.requests, w.block_table, cfg_for(w), B.options(**opts))
    inf = hp.info.as_dict()
    hp.close()
    return inf


@pytest.mark.parametrize("kv,build", [(7 * 128, 0), (8 * 128, 1), (8 * 128 + 1, 1),
                                      (4 * 128, 0)])
def test_copies_build_from_8_key_tiles(L, kv, build):
    # one-row CTAs (MHA decodes): the build that spreads a row's keys over 4
    # copies is chosen when most key tiles sit in CTAs of >= 8 tiles of 128
    inf = _host_info([(1, kv)] * 3, dict(kv_chunk=8192), n_q_heads=4, n_kv_heads=4,
                     head_dim=128, page_size=16)
    assert inf["n_decode_items"] == 3 * 4
    assert inf["splitkv_copies"] == build


def test_copies_build_needs_at_most_32_rows(L):
    # 48 rows per CTA (12 new rows x 4 query heads): one thread per row
    inf = _host_info([(12, 4000)], dict(kv_chunk=8192, prefill_min_rows=-1), n_q_heads=8,
                     n_kv_heads=2, head_dim=128, page_size=64)
    assert inf["splitkv_max_rows"] == 48 and inf["splitkv_copies"] == 0


@pytest.mark.parametrize("name,rows", [("decode_heavy_gqa4", 4), ("spec_decode_k3", 16),
                                       ("shared_prefix_decode", 24),
                                       ("llama2_7b_orca_iteration", 1)])
def test_plan_reports_largest_splitkv_cta(L, name, rows):
    # the rows of one split-KV CTA: a decode's g = 4 query heads; a speculative
    # step's (k + 1) g; the 6 sharers x g of a cascade group; one MHA decode row
    w = W.make_workload(name, with_values=False)
    inf = B.HostPlan(w.requests, w.block_table, cfg_for(w)).info
    assert inf.splitkv_max_rows == rows


def test_prefill_tiles_skip_masked_tiles(L):
    # one 4096-row prefill: CTA t owns rows [256 t, 256 t + 256) and visits
    # exactly the 2 t + 2 KV tiles of 128 keys its last row can see
    w = W.make_workload("llama2_7b_orca_iteration", with_values=False)
    hp = B.HostPlan(w.requests, w.block_table, cfg_for(w))
    _, _, pitems, _ = decode_plan(hp)
    a = pitems[pitems["req"] == 0]
    assert len(a) == 32 * 16
    assert sorted(set((2 * (a["i0"] // 256) + 2 - a["n_kv_tiles"]).tolist())) == [0]
    # heaviest first
    assert np.all(np.diff(pitems["n_kv_tiles"]) <= 0)


@pytest.mark.parametrize("name", W.ORDER)
def test_append_targets_are_private_pages_in_every_workload(L, name):
    w = W.make_workload(name, with_values=False)
    assert B.check_append_targets(w.requests, w.block_table, cfg_for(w)) == (B.MB_OK, -1)


def test_append_into_a_shared_page_is_flagged(L):
    # requests 0 and 1 share page 5 as their first block; request 1's new row
    # (position 10 of page 5, page size 16) would be written into it
    reqs = np.array([[0, 1, 20], [1, 2, 11], [2, 3, 40]], np.int32)
    bt = np.array([[5, 6, 0], [5, 9, 0], [1, 2, 3]], np.int32)
    cfg = B.config(4, 2, 64, 16, 10, 3, 0.0)
    assert B.check_append_targets(reqs, bt, cfg) == (B.MB_ERR_SHARED_PAGE, 1)
    # request 1 now appends at position 16 (page 9, its own): fine; request 0's
    # new row at 19 is in page 6, also its own
    reqs[1] = [1, 2, 17]
    assert B.check_append_targets(reqs, bt, cfg) == (B.MB_OK, -1)
    # a page mapped twice by the same request counts as one mapping
    bt2 = bt.copy()
    bt2[2] = [1, 1, 3]
    reqs2 = np.array([[0, 1, 20], [1, 2, 17], [2, 3, 20]], np.int32)
    assert B.check_append_targets(reqs2, bt2, cfg) == (B.MB_OK, -1)
    # only a shared page that receives a row counts: request 0 maps page 5 but
    # appends nothing; request 2 maps it too and appends into page 3
    reqs4 = np.array([[0, 0, 16], [0, 1, 11], [1, 2, 40]], np.int32)
    bt4 = np.array([[5, 0, 0], [6, 0, 0], [5, 7, 3]], np.int32)
    assert B.check_append_targets(reqs4, bt4, cfg) == (B.MB_OK, -1)


# ---------------------------------------------------------------- rotary helpers

def test_rope_table_matches_oracle(L):
    from oracle import rope as OR
    for d, base, pmax in [(128, 10000.0, 40000), (64, 10000.0, 300), (128, 500000.0, 1000)]:
        got = B.rope_table(pmax, d, base)
        ref = OR.table(pmax, d, base)
        # one rounding of an fp64 value to fp32: |err| <= 2^-24 * |value| <= 6e-8
        np.testing.assert_allclose(got.astype(np.float64), ref, rtol=0, atol=1.2e-7)
    out = np.empty((2, 8), np.float32)
    assert L.mb_rope_table(out.ctypes.data, 2, 7, ctypes.c_float(10000.0)) == MB_ERR_INVALID_ARG
    assert L.mb_rope_table(out.ctypes.data, 0, 8, ctypes.c_float(10000.0)) == MB_ERR_INVALID_ARG
    assert L.mb_rope_table(None, 2, 8, ctypes.c_float(10000.0)) == MB_ERR_INVALID_ARG


def test_positions_follow_the_triples(L):
    reqs = np.array([[0, 3, 10], [3, 3, 5], [5, 6, 1], [6, 10, 4]], np.int32)
    got = B.positions(reqs, 11)
    np.testing.assert_array_equal(got, [7, 8, 9, -1, -1, 0, 0, 1, 2, 3, -1])
    bad = np.array([[0, 3, 2]], np.int32)  # q_rows > kv_length
    out = np.empty(3, np.int32)
    assert L.mb_positions(bad.ctypes.data, 1, out.ctypes.data, 3) == MB_ERR_SHAPE

# ctypes mirrors of the public structs against the C headers, field by field
_MIRRORS = [("mb_request_t", "Request"), ("mb_config_t", "Config"),
            ("mb_plan_options_t", "PlanOptions"), ("mb_plan_info_t", "PlanInfo"),
            ("mb_sched_config_t", "SchedConfig"), ("mb_sched_stats_t", "SchedStats")]


def test_binding_structs_match_the_headers(tmp_path):
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda_inc = next((d for d in ("/usr/local/cuda/include",
                                 os.path.join(os.environ.get("CUDA_HOME", ""), "include"))
                     if d and os.path.exists(os.path.join(d, "cuda_runtime_api.h"))), None)
    if cc is None or cuda_inc is None:
        pytest.skip("no C compiler or CUDA headers")
    lines = []
    for c_name, py_name in _MIRRORS:
        cls = getattr(B, py_name)
        lines.append(f'  printf("{py_name} size %zu\\n", sizeof({c_name}));')
        for f, _ in cls._fields_:
            lines.append(f'  printf("{py_name} {f} %zu\\n", offsetof({c_name}, {f}));')
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "mb.h"\n#include "mb_sched.h"\n'
                   "int main(void) {\n" + "\n".join(lines) + "\n  return 0;\n}\n")
    exe = tmp_path / "layout"
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    subprocess.run([cc, "-std=c11", "-I", os.path.join(root, "include"), "-I", cuda_inc,
                    str(src), "-o", str(exe)], check=True, capture_output=True)
    got = {}
    for ln in subprocess.run([str(exe)], check=True, capture_output=True,
                             text=True).stdout.splitlines():
        name, field, val = ln.split()
        got[(name, field)] = int(val)
    for _, py_name in _MIRRORS:
        cls = getattr(B, py_name)
        assert got[(py_name, "size")] == ctypes.sizeof(cls), py_name
        for f, _ in cls._fields_:
            assert got[(py_name, f)] == getattr(cls, f).offset, (py_name, f)
