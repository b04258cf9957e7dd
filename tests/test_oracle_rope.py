"""Pins of the rotary-embedding oracle (``oracle/rope.py``), CPU only.

The pages name the fused "norm + RoPE + write KV" kernel without printing the
rotation, so nothing here comes from a printed value: every pin is fixed by
the mathematics of the reading documented in the oracle -- a rotation of each
(x_i, x_{i + D/2}) pair by a position-linear angle whose frequencies form the
geometric schedule from 1 down to 1/base:

* the same rotation written as complex multiplication by exp(i * angle);
* position 0 is the identity, norms are preserved, and a dot product of a
  rotated query and key depends only on their position difference;
* the angle table obeys the addition theorem row by row;
* the fused append writes exactly the rotated K and the unchanged V at each
  token's slot and nothing else.

Planted mistakes (pairing, rotation direction, frequency exponent, position
offset, unrotated K) each fail at least one pin.
"""

import math

import numpy as np
import pytest

from oracle import rope as R

RNG = np.random.default_rng(11)


def check_frequencies():
    for d, base in [(8, 10000.0), (64, 10000.0), (128, 10000.0), (128, 500000.0)]:
        th = R.inverse_frequencies(d, base)
        assert th.shape == (d // 2,)
        assert th[0] == 1.0
        ratios = th[1:] / th[:-1]
        np.testing.assert_allclose(ratios, ratios[0], rtol=1e-12)
        # geometric from 1 towards 1/base: D/2 steps of the ratio reach 1/base
        np.testing.assert_allclose(ratios[0] ** (d // 2), 1.0 / base, rtol=1e-10)


def check_position_zero_identity():
    x = RNG.standard_normal((5, 3, 16))
    tab = R.table(4, 16)
    np.testing.assert_array_equal(R.rotate(x, np.zeros(5, int), tab), x)


def check_complex_form():
    d = 32
    x = RNG.standard_normal((7, 2, d))
    pos = np.array([0, 1, 2, 17, 100, 999, 4095])
    tab = R.table(4096, d)
    got = R.rotate(x, pos, tab)
    z = x[..., : d // 2] + 1j * x[..., d // 2:]
    a = R.angles(pos, d)[:, None, :]
    zr = z * np.exp(1j * a)
    np.testing.assert_allclose(got[..., : d // 2], zr.real, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got[..., d // 2:], zr.imag, rtol=0, atol=1e-12)


def check_norm_and_relative_position():
    d = 64
    tab = R.table(3000, d)
    q = RNG.standard_normal((1, 1, d))
    k = RNG.standard_normal((1, 1, d))
    # every (x_i, x_{i + D/2}) pair keeps its length
    xr = R.rotate(q, [1234], tab)
    np.testing.assert_allclose(q[..., :32] ** 2 + q[..., 32:] ** 2,
                               xr[..., :32] ** 2 + xr[..., 32:] ** 2, rtol=1e-12)
    # <R(p) q, R(s) k> depends on p - s only
    for p, s in [(5, 2), (300, 17), (2000, 1999)]:
        ref = float((R.rotate(q, [p], tab) * R.rotate(k, [s], tab)).sum())
        for c in (1, 7, 250, 999 - s if 999 > s else 0):
            if p + c < 3000 and s + c < 3000:
                v = float((R.rotate(q, [p + c], tab) * R.rotate(k, [s + c], tab)).sum())
                assert math.isclose(v, ref, rel_tol=1e-9, abs_tol=1e-9)


def check_table_addition_theorem():
    d = 16
    tab = R.table(256, d)
    half = d // 2
    c, s = tab[:, :half], tab[:, half:]
    np.testing.assert_array_equal(tab[0], np.r_[np.ones(half), np.zeros(half)])
    np.testing.assert_allclose(c ** 2 + s ** 2, 1.0, rtol=1e-12)
    # row 1 holds the base angles themselves
    np.testing.assert_allclose(np.arctan2(s[1], c[1]), R.inverse_frequencies(d), rtol=1e-12)
    for p, q in [(1, 1), (3, 9), (100, 155)]:
        np.testing.assert_allclose(c[p + q], c[p] * c[q] - s[p] * s[q], atol=1e-12)
        np.testing.assert_allclose(s[p + q], s[p] * c[q] + c[p] * s[q], atol=1e-12)


def check_fused_append():
    ps, pages, hkv, hq, d = 4, 6, 2, 4, 8
    t = 5
    tab = R.table(64, d)
    q = RNG.standard_normal((t, hq, d))
    kn = RNG.standard_normal((t, hkv, d))
    vn = RNG.standard_normal((t, hkv, d))
    pos = np.array([3, 4, 9, 0, 63])
    slots = np.array([5, 6, -1, 22, 0])
    sentinel = 123.0
    kc = np.full((pages, hkv, ps, d), sentinel)
    vc = np.full((pages, hkv, ps, d), sentinel)
    qr, kc, vc = R.rope_kv_append(q, kc, vc, kn, vn, pos, slots, tab, ps)
    np.testing.assert_allclose(qr, R.rotate(q, pos, tab), rtol=0, atol=0)
    written = set()
    for i, slot in enumerate(slots.tolist()):
        if slot < 0:
            continue
        page, off = slot // ps, slot % ps
        written.add((page, off))
        # K: the complex-form rotation of the token's k at its position
        z = kn[i, :, : d // 2] + 1j * kn[i, :, d // 2:]
        zr = z * np.exp(1j * R.angles([pos[i]], d)[0])
        np.testing.assert_allclose(kc[page, :, off, : d // 2], zr.real, atol=1e-12)
        np.testing.assert_allclose(kc[page, :, off, d // 2:], zr.imag, atol=1e-12)
        np.testing.assert_array_equal(vc[page, :, off], vn[i])
    for page in range(pages):
        for off in range(ps):
            if (page, off) not in written:
                assert np.all(kc[page, :, off] == sentinel) and np.all(vc[page, :, off] == sentinel)


PIN_CHECKS = [check_frequencies, check_position_zero_identity, check_complex_form,
              check_norm_and_relative_position, check_table_addition_theorem, check_fused_append]


@pytest.mark.parametrize("check", PIN_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check()


# ------------------------------------------------------------------ mutants

def _rotate_interleaved(x, positions, cos_sin):
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    rows = np.asarray(cos_sin, dtype=np.float64)[np.asarray(positions, dtype=np.int64)]
    c, s = rows[:, None, : d // 2], rows[:, None, d // 2:]
    out = np.empty_like(x)
    out[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
    out[..., 1::2] = x[..., 1::2] * c + x[..., 0::2] * s
    return out


def _wrap_rotate_sign(orig):
    def rotate(x, positions, cos_sin):
        tab = np.asarray(cos_sin, dtype=np.float64).copy()
        tab[:, tab.shape[1] // 2:] *= -1
        return orig(x, positions, tab)
    return rotate


def _wrap_rotate_position_plus_one(orig):
    def rotate(x, positions, cos_sin):
        return orig(x, np.asarray(positions) + 1, cos_sin)
    return rotate


def _inv_freq_wrong_exponent(head_dim, base=10000.0):
    i = np.arange(head_dim // 2, dtype=np.float64)
    return base ** (-1.0 * i / head_dim)


def _wrap_append_unrotated_k(orig):
    def fused(q, k_cache, v_cache, k_new, v_new, positions, slots, cos_sin, page_size):
        qr, kc, vc = orig(q, k_cache, v_cache, k_new, v_new, positions, slots, cos_sin, page_size)
        for t, slot in enumerate(np.asarray(slots).tolist()):
            if slot >= 0:
                kc[slot // page_size, :, slot % page_size, :] = k_new[t]
        return qr, kc, vc
    return fused


MUTANTS = {
    "pairs_interleaved": ("rotate", lambda orig: _rotate_interleaved),
    "rotation_direction": ("rotate", _wrap_rotate_sign),
    "position_off_by_one": ("rotate", _wrap_rotate_position_plus_one),
    "frequency_exponent": ("inverse_frequencies", lambda orig: _inv_freq_wrong_exponent),
    "k_not_rotated": ("rope_kv_append", _wrap_append_unrotated_k),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, monkeypatch):
    attr, make = MUTANTS[name]
    monkeypatch.setattr(R, attr, make(getattr(R, attr)))
    caught = []
    for check in PIN_CHECKS:
        try:
            check()
        except (AssertionError, IndexError, ValueError):
            caught.append(check.__name__)
    assert caught, f"planted mistake {name} passed every pin"
