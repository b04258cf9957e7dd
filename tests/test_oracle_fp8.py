"""Pins of the fp8 (e4m3) cache oracle (``oracle/fp8.py``), CPU only.

* the codec against the format's definition (code 0x38 = 1, 0x7E = 448, the
  smallest subnormal 2^-9 = 0x01, the smallest normal 2^-6 = 0x08, strictly
  increasing magnitudes) and against a library routine, torch's
  float8_e4m3fn conversion, on random values inside the finite range;
* round to nearest with ties to the even code, saturation at 448;
* per-row quantization: the row's largest magnitude lands on +-448 exactly,
  every value comes back within half a unit of e4m3 precision, zero rows give
  zero codes and scale 0;
* the fp8 append writes codes and scales at the token's slot and nowhere else.
Planted mistakes (ties away from zero, the e5m2 maximum, a per-tensor scale,
lost signs) each fail at least one pin.
"""

import numpy as np
import pytest
import torch

from oracle import fp8 as F

RNG = np.random.default_rng(5)


def check_codec_definition():
    v = F.decode(np.arange(256, dtype=np.uint8))
    assert v[0x38] == 1.0 and v[0x7E] == 448.0 and v[0x01] == 2.0 ** -9
    assert v[0x08] == 2.0 ** -6 and v[0x07] == 7 * 2.0 ** -9
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    pos = v[:127]
    assert np.all(np.diff(pos) > 0)
    np.testing.assert_array_equal(v[0x80:0xFF], -pos)
    # every finite code round-trips
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    np.testing.assert_array_equal(F.encode(F.decode(codes)), codes)


def check_codec_against_library():
    x = np.concatenate([RNG.standard_normal(20000) * s for s in (1e-3, 0.1, 1, 30, 300)])
    x = x[np.abs(x) <= 440].astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(F.encode(x), ref)


def check_rounding_rules():
    v = F.decode(np.arange(127, dtype=np.uint8))
    mids = (v[:-1] + v[1:]) / 2
    got = F.encode(mids)
    lo = np.arange(126)
    want = np.where(lo % 2 == 0, lo, lo + 1)          # the even code
    np.testing.assert_array_equal(got, want.astype(np.uint8))
    np.testing.assert_array_equal(F.encode(np.array([449.0, 1e6, -500.0])),
                                  np.array([0x7E, 0x7E, 0xFE], np.uint8))


def check_row_quantization():
    x = (RNG.standard_normal((300, 128)) * RNG.choice([1e-3, 1, 50], size=(300, 1))).astype(np.float32)
    codes, scales = F.quantize_rows(x)
    assert codes.dtype == np.uint8 and scales.dtype == np.float32
    deq = F.dequantize_rows(codes, scales)
    amax_code = np.max(np.abs(F.decode(codes)), axis=1)
    np.testing.assert_array_equal(amax_code, 448.0)
    # half an e4m3 unit: 2^-4 relative for normal values, 2^-10 * scale below
    bound = np.maximum(np.abs(x) * 2.0 ** -4, scales[:, None].astype(np.float64) * 2.0 ** -10)
    assert np.all(np.abs(deq - x) <= bound * (1 + 1e-6))
    z_codes, z_scales = F.quantize_rows(np.zeros((2, 64), np.float32))
    assert np.all(z_codes == 0) and np.all(z_scales == 0)


def check_append():
    ps, pages, hkv, d = 4, 5, 2, 8
    k8 = np.full((pages, hkv, ps, d), 0xAA, np.uint8)
    v8 = k8.copy()
    ks = np.full((pages, hkv, ps), -1.0, np.float32)
    vs = ks.copy()
    kn = RNG.standard_normal((3, hkv, d)).astype(np.float32)
    vn = RNG.standard_normal((3, hkv, d)).astype(np.float32)
    slots = np.array([6, -1, 17])
    F.append_scatter_fp8(k8, v8, ks, vs, kn, vn, slots, ps)
    for t, slot in [(0, 6), (2, 17)]:
        p, o = divmod(slot, ps)
        c, s = F.quantize_rows(kn[t])
        np.testing.assert_array_equal(k8[p, :, o], c)
        np.testing.assert_array_equal(ks[p, :, o], s)
        c, s = F.quantize_rows(vn[t])
        np.testing.assert_array_equal(v8[p, :, o], c)
        np.testing.assert_array_equal(vs[p, :, o], s)
    written = {(1, 2), (4, 1)}
    for p in range(pages):
        for o in range(ps):
            if (p, o) not in written:
                assert np.all(k8[p, :, o] == 0xAA) and np.all(ks[p, :, o] == -1.0)


PIN_CHECKS = [check_codec_definition, check_codec_against_library, check_rounding_rules,
              check_row_quantization, check_append]


@pytest.mark.parametrize("check", PIN_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check()


def _encode_ties_away(orig):
    def encode(x):
        x = np.asarray(x, dtype=np.float64)
        a = np.minimum(np.abs(x), F.E4M3_MAX)
        lo = np.searchsorted(F._POS, a, side="right") - 1
        hi = np.minimum(lo + 1, 126)
        code = np.where((F._POS[hi] - a) <= (a - F._POS[lo]), hi, lo).astype(np.uint8)
        return code | (np.signbit(x).astype(np.uint8) << 7)
    return encode


def _quantize_e5m2_max(orig):
    def quantize_rows(x):
        x32 = np.asarray(x, dtype=np.float32)
        scale = (np.max(np.abs(x32), axis=-1) / np.float32(57344.0)).astype(np.float32)
        safe = np.where(scale > 0, scale, np.float32(1)).astype(np.float32)
        return F.encode((x32 / safe[..., None]).astype(np.float32)), scale
    return quantize_rows


def _quantize_per_tensor(orig):
    def quantize_rows(x):
        x32 = np.asarray(x, dtype=np.float32)
        s = np.float32(np.max(np.abs(x32)) / np.float32(448.0))
        scale = np.full(x32.shape[:-1], s, np.float32)
        return F.encode((x32 / s).astype(np.float32)), scale
    return quantize_rows


def _encode_unsigned(orig):
    def encode(x):
        return orig(np.abs(np.asarray(x, dtype=np.float64)))
    return encode


MUTANTS = {
    "ties_away_from_zero": ("encode", _encode_ties_away),
    "e5m2_maximum": ("quantize_rows", _quantize_e5m2_max),
    "per_tensor_scale": ("quantize_rows", _quantize_per_tensor),
    "sign_lost": ("encode", _encode_unsigned),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, monkeypatch):
    attr, make = MUTANTS[name]
    monkeypatch.setattr(F, attr, make(getattr(F, attr)))
    caught = []
    for check in PIN_CHECKS:
        try:
            check()
        except (AssertionError, IndexError, ValueError):
            caught.append(check.__name__)
    assert caught, f"planted mistake {name} passed every pin"
