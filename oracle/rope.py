"""NumPy fp64 oracle for the rotary position embedding fused into the KV
append (the step just before the attention reads the cache).

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

What is computed, and where it comes from
-----------------------------------------
* "GLM-5.3 e2e token ledger", the per-layer forward (stage 6) and its fusion
  table: the norm, RoPE and the KV write run as one fused kernel that already
  holds the layer's q and k, so writing K into the cache costs no extra pass.
  The pages name RoPE without defining it. The reading taken here is the
  rotary embedding of the Llama-2 family the other pages use: for a head
  vector x of even length D at position p, the pairs (x_i, x_{i + D/2}),
  i < D/2, are rotated by the angle p * base^(-2 i / D) (base 10000):
      x'_i         = x_i cos(a) - x_{i+D/2} sin(a)
      x'_{i + D/2} = x_{i+D/2} cos(a) + x_i sin(a).
  Q and K are rotated at their token's position; V is not; the cache then
  receives the rotated K and the plain V at the token's slot (the append of
  "ORCA and chunked prefill", section 4).
* The angle table ``cos_sin[p] = [cos(p theta_0..theta_{D/2-1}),
  sin(p theta_0..)]`` is an input of the fused operation (the caller builds
  it once per model); ``table`` builds it here in fp64 from the definition.
"""

from __future__ import annotations

import numpy as np


def inverse_frequencies(head_dim: int, base: float = 10000.0) -> np.ndarray:
    """theta_i = base^(-2 i / D), i < D/2 (fp64)."""
    if head_dim % 2:
        raise ValueError("head_dim must be even")
    i = np.arange(head_dim // 2, dtype=np.float64)
    return base ** (-2.0 * i / head_dim)


def angles(positions, head_dim: int, base: float = 10000.0) -> np.ndarray:
    """[len(positions), D/2] angles p * theta_i in fp64."""
    p = np.asarray(positions, dtype=np.float64).reshape(-1, 1)
    return p * inverse_frequencies(head_dim, base)[None, :]


def table(max_position: int, head_dim: int, base: float = 10000.0) -> np.ndarray:
    """[max_position, D] fp64: cos of the D/2 angles, then their sin."""
    a = angles(np.arange(max_position), head_dim, base)
    return np.concatenate([np.cos(a), np.sin(a)], axis=1)


def rotate(x: np.ndarray, positions, cos_sin: np.ndarray) -> np.ndarray:
    """Rotate every head vector of ``x`` [T, H, D] at its token's position.

    ``cos_sin`` is a table as built by ``table`` (any precision; used as
    given, upcast to fp64). Returns fp64 [T, H, D].
    """
    x = np.asarray(x, dtype=np.float64)
    t, h, d = x.shape
    half = d // 2
    rows = np.asarray(cos_sin, dtype=np.float64)[np.asarray(positions, dtype=np.int64)]
    c = rows[:, None, :half]
    s = rows[:, None, half:]
    lo, hi = x[..., :half], x[..., half:]
    out = np.empty_like(x)
    out[..., :half] = lo * c - hi * s
    out[..., half:] = hi * c + lo * s
    return out


def rope_kv_append(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray,
                   v_new: np.ndarray, positions, slots, cos_sin: np.ndarray, page_size: int):
    """The fused operation: rotated Q (returned, fp64), rotated K written into
    ``k_cache`` (fp64 array [pages, Hkv, ps, D]) and V (copied as given) into
    ``v_cache`` at each token's slot; a negative slot skips the token's K/V.
    Returns (q_rot, k_cache, v_cache)."""
    q_rot = rotate(q, positions, cos_sin)
    k_rot = rotate(k_new, positions, cos_sin)
    for t, slot in enumerate(np.asarray(slots).tolist()):
        if slot < 0:
            continue
        page, off = divmod(int(slot), page_size)
        k_cache[page, :, off, :] = k_rot[t]
        v_cache[page, :, off, :] = np.asarray(v_new[t], dtype=k_cache.dtype)
    return q_rot, k_cache, v_cache
