"""Pure-Python brute-force attention for tiny inputs.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The same definition as ``oracle.attention.attend`` written with nested loops,
Python floats and ``math.exp``/``math.log``, no NumPy. It exists to pin the
NumPy oracle: the two are written independently and must agree to ~1e-12.

Definition followed ("How To Scale Your Model notes (7-8)", §2; "One forward,
many requests", §6.2; "LLM end to end", §4-§6): for new row ``i`` of ``m``
with ``S0 = kv - m`` cached columns, column ``j`` is visible iff
``j <= S0 + i``; score ``s_ij = scale * sum_d q_id k_jd``; weights are the
softmax over the visible columns; output row is the weighted sum of V rows.
Query head ``h`` uses KV head ``h // (Hq // Hkv)``.
"""

from __future__ import annotations

import math


def attend(q, k, v, scale=None):
    """q: nested lists ``[m][Hq][D]``; k, v: ``[kv][Hkv][D]``.

    Returns ``(out [m][Hq][D], lse [m][Hq])`` as nested lists of floats.
    """
    m = len(q)
    hq = len(q[0])
    d = len(q[0][0])
    kv = len(k)
    hkv = len(k[0])
    g = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    s0 = kv - m
    out = [[[0.0] * d for _ in range(hq)] for _ in range(m)]
    lse = [[0.0] * hq for _ in range(m)]
    for i in range(m):
        last = s0 + i  # last visible column (inclusive)
        for h in range(hq):
            kh = h // g
            scores = []
            for j in range(last + 1):
                acc = 0.0
                for c in range(d):
                    acc += float(q[i][h][c]) * float(k[j][kh][c])
                scores.append(acc * scale)
            mx = max(scores)
            ex = [math.exp(s - mx) for s in scores]
            z = sum(ex)
            for c in range(d):
                acc = 0.0
                for j in range(last + 1):
                    acc += ex[j] * float(v[j][kh][c])
                out[i][h][c] = acc / z
            lse[i][h] = mx + math.log(z)
    return out, lse
