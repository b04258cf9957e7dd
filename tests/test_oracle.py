"""Pins for the CPU oracle (no GPU).

The oracle is trusted only because these tests tie it to facts outside
itself: the pages' worked example, special cases that reduce to library
routines, closed forms, invariants the pages state, and a brute force written
separately. A planted mistake in the oracle must fail at least one of them
(``test_planted_mistakes_are_caught``).
"""

import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import attention as A
from oracle import brute as B
from tests.conftest import read_int_table

RNG = np.random.default_rng(1234)


def rand(*shape, rng=RNG):
    return rng.standard_normal(shape)


def sdpa(q, k, v, scale, causal=False, mask=None):
    """torch SDPA in fp64 on CPU, GQA via enable_gqa. q [m,Hq,D], k/v [kv,Hkv,D]."""
    tq = torch.from_numpy(np.ascontiguousarray(q.transpose(1, 0, 2)))[None]
    tk = torch.from_numpy(np.ascontiguousarray(k.transpose(1, 0, 2)))[None]
    tv = torch.from_numpy(np.ascontiguousarray(v.transpose(1, 0, 2)))[None]
    am = None if mask is None else torch.from_numpy(mask)
    o = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=am, is_causal=causal, scale=scale,
        enable_gqa=(q.shape[1] != k.shape[1]))
    return o[0].numpy().transpose(1, 0, 2)


# --------------------------------------------------------------------------
# pin checks as plain functions, so the planted-mistake test can rerun them
# --------------------------------------------------------------------------

def check_worked_example():
    """How To Scale Your Model notes (7-8), section 2: cache abc + suffix xefg."""
    golden = np.array(read_int_table("abc_xefg_visibility.txt"), dtype=bool)
    assert golden.shape == (4, 7)
    vis = A.visible(3, 4)
    assert vis.shape == (4, 7)
    assert np.array_equal(vis, golden)
    assert int((~golden).sum()) == 6
    rng = np.random.default_rng(7)
    q, k, v = rand(4, 2, 8, rng=rng), rand(7, 1, 8, rng=rng), rand(7, 1, 8, rng=rng)
    _, _, w = A.attend(q, k, v, None, return_weights=True)
    assert w.shape == (2, 4, 7)
    for h in range(2):
        assert np.all(w[h][~golden] == 0.0)
        assert np.all(w[h][golden] > 0.0)
        np.testing.assert_allclose(w[h].sum(axis=1), 1.0, rtol=0, atol=1e-14)


def check_brute_force():
    rng = np.random.default_rng(11)
    for (m, kv, hq, hkv, d) in [(1, 1, 1, 1, 4), (3, 3, 2, 1, 4), (4, 7, 4, 2, 8),
                                (1, 9, 2, 2, 3), (5, 12, 6, 3, 5), (2, 20, 4, 1, 8)]:
        q, k, v = rand(m, hq, d, rng=rng), rand(kv, hkv, d, rng=rng), rand(kv, hkv, d, rng=rng)
        scale = 0.37 if d == 5 else None
        o, l = A.attend(q, k, v, scale)
        ob, lb = B.attend(q.tolist(), k.tolist(), v.tolist(), scale)
        np.testing.assert_allclose(o, np.array(ob), rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, np.array(lb), rtol=0, atol=1e-12)


def check_decode_special_case():
    """m = 1: a single unmasked softmax over all kv columns (library SDPA)."""
    rng = np.random.default_rng(12)
    for (kv, hq, hkv, d) in [(1, 2, 1, 8), (33, 4, 2, 16), (200, 8, 2, 64)]:
        q, k, v = rand(1, hq, d, rng=rng), rand(kv, hkv, d, rng=rng), rand(kv, hkv, d, rng=rng)
        o, _ = A.attend(q, k, v)
        ref = sdpa(q, k, v, 1.0 / math.sqrt(d))
        np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)


def check_full_prefill_special_case():
    """S0 = 0: textbook causal attention (library SDPA, is_causal)."""
    rng = np.random.default_rng(13)
    for (m, hq, hkv, d) in [(1, 1, 1, 4), (17, 4, 2, 16), (64, 4, 1, 32)]:
        q, k, v = rand(m, hq, d, rng=rng), rand(m, hkv, d, rng=rng), rand(m, hkv, d, rng=rng)
        o, _ = A.attend(q, k, v)
        ref = sdpa(q, k, v, 1.0 / math.sqrt(d), causal=True)
        np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)


def check_general_vs_library_softmax():
    """Any S0, m: library SDPA with the visibility mask, and lse vs logsumexp."""
    rng = np.random.default_rng(14)
    for (m, kv, hq, hkv, d, scale) in [(4, 7, 2, 1, 8, None), (9, 40, 6, 2, 16, 0.21),
                                       (32, 160, 4, 2, 64, 0.125)]:
        q, k, v = rand(m, hq, d, rng=rng), rand(kv, hkv, d, rng=rng), rand(kv, hkv, d, rng=rng)
        o, l = A.attend(q, k, v, scale)
        sc = 1.0 / math.sqrt(d) if scale is None else scale
        ref = sdpa(q, k, v, sc, mask=A.visible(kv - m, m))
        np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)
        g = hq // hkv
        vis = A.visible(kv - m, m)
        for h in range(hq):
            s = (q[:, h] @ k[:, h // g].T) * sc
            s = np.where(vis, s, -np.inf)
            np.testing.assert_allclose(l[:, h], scipy.special.logsumexp(s, axis=1),
                                       rtol=1e-13, atol=1e-13)


def check_kv_one():
    """kv = 1 (a first prefill row): the output is v_0."""
    rng = np.random.default_rng(15)
    q, k, v = rand(1, 4, 8, rng=rng), rand(1, 2, 8, rng=rng), rand(1, 2, 8, rng=rng)
    o, l = A.attend(q, k, v)
    for h in range(4):
        np.testing.assert_array_equal(o[0, h], v[0, h // 2])
        np.testing.assert_allclose(l[0, h], (q[0, h] @ k[0, h // 2]) / math.sqrt(8), rtol=1e-15)


def check_closed_forms():
    rng = np.random.default_rng(16)
    m, kv, hq, hkv, d = 5, 11, 4, 2, 8
    s0 = kv - m
    q, v = rand(m, hq, d, rng=rng), rand(kv, hkv, d, rng=rng)
    # all keys equal -> uniform weights over the visible columns -> mean of visible V
    k_same = np.broadcast_to(rand(1, hkv, d, rng=rng), (kv, hkv, d)).copy()
    o, _ = A.attend(q, k_same, v)
    for i in range(m):
        for h in range(hq):
            np.testing.assert_allclose(o[i, h], v[: s0 + i + 1, h // 2].mean(axis=0),
                                       rtol=1e-12, atol=1e-12)
    # q = 0 -> uniform as well
    o0, l0 = A.attend(np.zeros((m, hq, d)), rand(kv, hkv, d, rng=rng), v)
    for i in range(m):
        np.testing.assert_allclose(o0[i, :, :], np.repeat(v[: s0 + i + 1].mean(axis=0), 2, axis=0),
                                   rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(l0[i], math.log(s0 + i + 1), rtol=1e-14)
    # constant V -> that constant
    vc = np.full((kv, hkv, d), 0.75)
    oc, _ = A.attend(q, rand(kv, hkv, d, rng=rng), vc)
    np.testing.assert_allclose(oc, 0.75, rtol=1e-13)


def check_chunked_equals_one_shot():
    """ORCA and chunked prefill, section 4: chunk k attends to the cached
    prefix without mask and to itself causally; the result equals the
    one-shot prefill."""
    rng = np.random.default_rng(17)
    n, hq, hkv, d = 37, 4, 2, 16
    q, k, v = rand(n, hq, d, rng=rng), rand(n, hkv, d, rng=rng), rand(n, hkv, d, rng=rng)
    full, lfull = A.attend(q, k, v)
    for chunks in ([10, 10, 10, 7], [1] * 37, [36, 1], [5, 32]):
        parts, lparts = [], []
        done = 0
        for c in chunks:
            o, l = A.attend(q[done:done + c], k[:done + c], v[:done + c])
            parts.append(o)
            lparts.append(l)
            done += c
        np.testing.assert_allclose(np.concatenate(parts), full, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(np.concatenate(lparts), lfull, rtol=1e-12, atol=1e-13)


def _paged_case(rng, perm_seed, ps=4, hq=4, hkv=2, d=8, shapes=((6, 6), (1, 9), (3, 10))):
    """Build caches with the oracle's scatter from logical K/V, pages permuted."""
    n = len(shapes)
    blocks = [math.ceil(kv / ps) for _, kv in shapes]
    pool = sum(blocks) + 3
    perm = np.random.default_rng(perm_seed).permutation(pool)
    bt = np.full((n, max(blocks)), -1, dtype=np.int64)
    cur = 0
    for r in range(n):
        bt[r, :blocks[r]] = perm[cur:cur + blocks[r]]
        cur += blocks[r]
    reqs = []
    qo = 0
    for q_rows, kv in shapes:
        reqs.append((qo, qo + q_rows, kv))
        qo += q_rows
    return reqs, bt, pool


def _fill(reqs, bt, pool, logical_k, logical_v, q_total, hkv, d, ps, sentinel=0.0):
    kc = np.full((pool, hkv, ps, d), sentinel)
    vc = np.full((pool, hkv, ps, d), sentinel)
    for r, (qs, qe, kv) in enumerate(reqs):
        for p in range(kv):
            page, slot = A.logical_position_location(bt[r], p, ps)
            kc[page, :, slot] = logical_k[r][p]
            vc[page, :, slot] = logical_v[r][p]
    return kc, vc


def check_page_permutation_and_isolation():
    """How To Scale Your Model notes (7-8), section 3: paging changes only the
    physical placement. One forward, many requests, section 6.2: each request
    reads only its own cache."""
    rng = np.random.default_rng(18)
    ps, hq, hkv, d = 4, 4, 2, 8
    shapes = ((6, 6), (1, 9), (3, 10))
    lk = [rand(kv, hkv, d, rng=rng) for _, kv in shapes]
    lv = [rand(kv, hkv, d, rng=rng) for _, kv in shapes]
    total_q = sum(q for q, _ in shapes)
    q = rand(total_q, hq, d, rng=rng)
    outs = []
    for seed in (0, 1, 2):
        reqs, bt, pool = _paged_case(rng, seed, ps, hq, hkv, d, shapes)
        kc, vc = _fill(reqs, bt, pool, lk, lv, total_q, hkv, d, ps)
        o, l = A.mixed_attention(q, kc, vc, reqs, bt, ps)
        outs.append((o, l))
        # request by request equals attend on the logical K/V
        for r, (qs, qe, kv) in enumerate(reqs):
            o_r, l_r = A.attend(q[qs:qe], lk[r], lv[r])
            np.testing.assert_array_equal(o[qs:qe], o_r)
            np.testing.assert_array_equal(l[qs:qe], l_r)
        # isolation: overwrite request 1's pages; requests 0 and 2 unchanged
        kc2, vc2 = kc.copy(), vc.copy()
        for b in range(math.ceil(shapes[1][1] / ps)):
            kc2[bt[1, b]] = 1e3
            vc2[bt[1, b]] = -1e3
        o2, _ = A.mixed_attention(q, kc2, vc2, reqs, bt, ps)
        qs1, qe1, _ = reqs[1]
        np.testing.assert_array_equal(o2[:qs1], o[:qs1])
        np.testing.assert_array_equal(o2[qe1:], o[qe1:])
        assert not np.allclose(o2[qs1:qe1], o[qs1:qe1])
        # pages outside every block table (sentinel pages) never matter
        unused = sorted(set(range(pool)) - set(bt[bt >= 0].tolist()))
        kc3, vc3 = kc.copy(), vc.copy()
        kc3[unused] = np.nan
        vc3[unused] = np.nan
        o3, _ = A.mixed_attention(q, kc3, vc3, reqs, bt, ps)
        np.testing.assert_array_equal(o3, o)
    for o, l in outs[1:]:
        np.testing.assert_array_equal(o, outs[0][0])
        np.testing.assert_array_equal(l, outs[0][1])


def check_heads_and_gqa_grouping():
    """LLM end to end, section 5: heads are independent. How To Scale Your
    Model notes (7-8), section 3: g query heads share a KV head (contiguous
    grouping: query head h reads KV head h // g)."""
    rng = np.random.default_rng(19)
    m, kv, hq, hkv, d = 3, 8, 6, 2, 8
    g = hq // hkv
    q, k, v = rand(m, hq, d, rng=rng), rand(kv, hkv, d, rng=rng), rand(kv, hkv, d, rng=rng)
    o, l = A.attend(q, k, v)
    # GQA equals MHA with each KV head repeated g times (repeat_interleave)
    o_mha, l_mha = A.attend(q, np.repeat(k, g, axis=1), np.repeat(v, g, axis=1))
    np.testing.assert_allclose(o, o_mha, rtol=0, atol=1e-15)
    np.testing.assert_allclose(l, l_mha, rtol=0, atol=1e-15)
    # head h alone equals a one-head problem on KV head h // g
    for h in range(hq):
        oh, lh = A.attend(q[:, h:h + 1], k[:, h // g:h // g + 1], v[:, h // g:h // g + 1])
        np.testing.assert_allclose(o[:, h:h + 1], oh, rtol=0, atol=1e-15)
    # perturbing one query head changes only that head
    q2 = q.copy()
    q2[:, 4] += 1.0
    o2, _ = A.attend(q2, k, v)
    mask = np.ones(hq, bool)
    mask[4] = False
    np.testing.assert_array_equal(o2[:, mask], o[:, mask])
    assert not np.allclose(o2[:, 4], o[:, 4])


def check_append_scatter():
    """Hand-worked addressing example (tests/golden/append_tiny.txt)."""
    rows = read_int_table("append_tiny.txt")
    ps, hkv, d = 4, 1, 2
    reqs = [(0, 3, 6), (3, 4, 9)]
    bt = np.array([[5, 2, -1], [0, 7, 4]])
    kc = np.zeros((8, hkv, ps, d), dtype=np.uint16)
    vc = np.zeros((8, hkv, ps, d), dtype=np.uint16)
    kn = (np.arange(4 * hkv * d, dtype=np.uint16).reshape(4, hkv, d) + 1)
    vn = kn + 100
    A.append_scatter(kc, vc, kn, vn, reqs, bt, ps)
    written = np.zeros((8, ps), bool)
    for t, page, slot, flat in rows:
        assert flat == page * ps + slot
        np.testing.assert_array_equal(kc[page, :, slot], kn[t])
        np.testing.assert_array_equal(vc[page, :, slot], vn[t])
        written[page, slot] = True
    kt, vt = kc.transpose(0, 2, 1, 3), vc.transpose(0, 2, 1, 3)
    assert np.all(kt[~written] == 0) and np.all(vt[~written] == 0)


PIN_CHECKS = [check_worked_example, check_brute_force, check_decode_special_case,
              check_full_prefill_special_case, check_general_vs_library_softmax,
              check_kv_one, check_closed_forms, check_chunked_equals_one_shot,
              check_page_permutation_and_isolation, check_heads_and_gqa_grouping,
              check_append_scatter]


@pytest.mark.parametrize("check", PIN_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check()


# --------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# --------------------------------------------------------------------------

def _mut_visible_no_diagonal(s0, m):
    vis = np.zeros((m, s0 + m), bool)
    vis[:, :s0] = True
    for i in range(m):
        vis[i, s0:s0 + i] = True
    vis[:, 0] = True  # keep rows non-empty so the mutant runs
    return vis


def _mut_visible_plus_one(s0, m):
    vis = np.zeros((m, s0 + m), bool)
    vis[:, :s0] = True
    for i in range(m):
        vis[i, s0:s0 + i + 2] = True
    return vis


def _mut_visible_prefix_causal(s0, m):
    # treats the cached prefix as causal to the rows (top-left alignment)
    vis = np.zeros((m, s0 + m), bool)
    for i in range(m):
        vis[i, :i + 1] = True
    return vis


def _mut_append_swap_page_slot(k_cache, v_cache, k_new, v_new, requests, block_table, page_size):
    for r, (qs, qe, kv) in enumerate(np.asarray(requests).tolist()):
        s0 = kv - (qe - qs)
        for t in range(qs, qe):
            p = s0 + (t - qs) + 1  # off by one position
            page = int(block_table[r][p // page_size])
            k_cache[page, :, p % page_size, :] = k_new[t]
            v_cache[page, :, p % page_size, :] = v_new[t]
    return k_cache, v_cache


def _wrap_attend_modulo_grouping(orig):
    def attend(q, k, v, scale=None, return_weights=False):
        hq, hkv = q.shape[1], k.shape[1]
        idx = np.arange(hq) % hkv
        return orig(q, np.asarray(k)[:, idx], np.asarray(v)[:, idx], scale, return_weights)
    return attend


def _wrap_attend_no_scale(orig):
    def attend(q, k, v, scale=None, return_weights=False):
        return orig(q, k, v, 1.0 if scale is None else scale, return_weights)
    return attend


def _wrap_attend_lse_without_max(orig):
    def attend(q, k, v, scale=None, return_weights=False):
        res = orig(q, k, v, scale, return_weights)
        res = list(res)
        res[1] = np.log(np.exp(res[1]) + 1e-3)
        return tuple(res)
    return attend


def _wrap_gather_transposed(orig):
    def gather(cache, bt_row, kv, ps):
        outv = np.empty((kv,) + cache.shape[1:2] + cache.shape[3:], dtype=cache.dtype)
        for p in range(kv):
            page = int(bt_row[p // ps])
            outv[p] = cache[page, :, (ps - 1 - p % ps), :]
        return outv
    return gather


MUTANTS = {
    "mask_drops_diagonal": ("visible", lambda orig: _mut_visible_no_diagonal),
    "mask_one_past_diagonal": ("visible", lambda orig: _mut_visible_plus_one),
    "mask_prefix_treated_causal": ("visible", lambda orig: _mut_visible_prefix_causal),
    "gqa_modulo_grouping": ("attend", _wrap_attend_modulo_grouping),
    "missing_softmax_scale": ("attend", _wrap_attend_no_scale),
    "lse_wrong": ("attend", _wrap_attend_lse_without_max),
    "append_off_by_one_position": ("append_scatter", lambda orig: _mut_append_swap_page_slot),
    "gather_slot_reversed": ("gather_logical", _wrap_gather_transposed),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, monkeypatch):
    attr, make = MUTANTS[name]
    orig = getattr(A, attr)
    monkeypatch.setattr(A, attr, make(orig))
    caught = []
    for check in PIN_CHECKS:
        try:
            check()
        except (AssertionError, IndexError, ValueError, FloatingPointError):
            caught.append(check.__name__)
    assert caught, f"planted mistake {name} passed every pin"


def test_oracle_imports_nothing_from_product():
    import ast
    import os
    root = os.path.dirname(oracle.__file__)
    for fn in os.listdir(root):
        if fn.endswith(".py"):
            tree = ast.parse(open(os.path.join(root, fn)).read())
            for node in ast.walk(tree):
                if isinstance(node, (ast.Import, ast.ImportFrom)):
                    names = [a.name for a in node.names] if isinstance(node, ast.Import) else [node.module or ""]
                    for n in names:
                        assert "continuous_batching_paged_varlen_gb300" not in n
                        assert n.split(".")[0] not in ("torch", "ctypes")
