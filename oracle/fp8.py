"""NumPy oracle for the fp8 (e4m3) KV cache variant.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

What is computed, and where it comes from
-----------------------------------------
* "GLM-5.3 e2e token ledger", the KV layout paragraphs: the cache stores K/V
  as FP8 with FP32 scales kept next to the data, one scale per 128 FP8 values
  (four scales for a 512-byte row), and a kernel must read both to
  dequantize. The reading taken for this GQA cache: e4m3 codes
  ``[pages, Hkv, ps, D]`` and one fp32 scale per (token, KV head) row of D
  values, ``scale = amax(|row|) / 448`` (448 = the largest finite e4m3
  value), ``code = e4m3(x / scale)`` rounded to nearest, ties to even,
  saturating at +-448; a row of zeros gets scale 0 and zero codes. The value
  a kernel reads back is ``decode(code) * scale``.
* Where floating point decides an integer (the codes), the oracle takes the
  decision in the product's precision: amax and the scale in fp32, the
  quotient ``x / scale`` as one IEEE fp32 division.
* Attention over an fp8 cache is the attention of ``oracle.attention`` on the
  dequantized K/V (fp64).

The e4m3 codec is written from the format's definition (1 sign bit, 4
exponent bits with bias 7, 3 mantissa bits, subnormals at exponent 0, no
infinities, S.1111.111 = NaN).
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def _e4m3_positive_values() -> np.ndarray:
    """The value of every code 0x00..0x7E (0x7F is NaN), fp64."""
    vals = np.empty(127, dtype=np.float64)
    for code in range(127):
        e, m = code >> 3, code & 7
        if e == 0:
            vals[code] = (m / 8.0) * 2.0 ** (1 - 7)       # subnormal
        else:
            vals[code] = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_POS = _e4m3_positive_values()


def decode(codes) -> np.ndarray:
    """uint8 e4m3 codes -> fp64 values (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes, dtype=np.uint8)
    mag = c & 0x7F
    out = np.where(mag == 0x7F, np.nan, _POS[np.minimum(mag, 126)])
    return np.where(c & 0x80, -out, out)


def encode(x) -> np.ndarray:
    """Finite values -> uint8 e4m3 codes: nearest value, ties to the even code
    (even mantissa), magnitudes beyond 448 saturate to 448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    # index of the largest code value <= a, and the one above
    lo = np.searchsorted(_POS, a, side="right") - 1
    hi = np.minimum(lo + 1, 126)
    dlo = a - _POS[lo]
    dhi = _POS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi != lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    # the sign survives rounding to zero (-0 is code 0x80), as in IEEE rounding
    sign = np.signbit(x).astype(np.uint8) << 7
    return code | sign


def quantize_rows(x) -> tuple[np.ndarray, np.ndarray]:
    """Per-row quantization of ``x`` [..., D] (bf16 values given as fp32 or
    fp64): returns (codes uint8 [..., D], scales fp32 [...])."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=-1)                       # exact in fp32
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)  # one fp32 division
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    q = (x32 / safe[..., None]).astype(np.float32)            # one fp32 division per value
    codes = encode(q)
    codes = np.where((scale > 0)[..., None], codes, np.uint8(0)).astype(np.uint8)
    return codes, scale


def dequantize_rows(codes, scales) -> np.ndarray:
    return decode(codes) * np.asarray(scales, dtype=np.float64)[..., None]


def append_scatter_fp8(k8, v8, ks, vs, k_new, v_new, slots, page_size):
    """Quantize each token's K/V rows and write codes and scales at its slot
    (negative slot: skipped). k8/v8 uint8 [pages, Hkv, ps, D], ks/vs fp32
    [pages, Hkv, ps]; k_new/v_new [T, Hkv, D] values. Returns the arrays."""
    kc, ksc = quantize_rows(k_new)
    vc, vsc = quantize_rows(v_new)
    for t, slot in enumerate(np.asarray(slots).tolist()):
        if slot < 0:
            continue
        page, off = divmod(int(slot), page_size)
        k8[page, :, off, :] = kc[t]
        v8[page, :, off, :] = vc[t]
        ks[page, :, off] = ksc[t]
        vs[page, :, off] = vsc[t]
    return k8, v8, ks, vs
