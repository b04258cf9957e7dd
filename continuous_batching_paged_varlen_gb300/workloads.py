"""Seeded synthetic inputs for the mixed-iteration attention step.

This module is shared by the tests, the bench and the CPU oracle's callers.
It holds no attention arithmetic and no cache addressing: it only draws the
request shapes, the page assignment (block tables) and the bf16 Q/K/V
values. Each request's K/V come out in *logical* order (history positions
``[0, S0)`` and this iteration's new rows); where they land in the paged
cache is decided elsewhere (by the library's slot mapping on the product
side, by the oracle's own gather/scatter on the test side).

The five workloads follow the shapes the pages use: a tiny mixed iteration;
the Llama-2-7B single-layer ORCA iteration of "ORCA and chunked prefill", §2
(a 4096-row prefill next to decodes of kv 1500 and 1700); a decode-heavy GQA
batch; a chunked-prefill chunk (2048 rows at S0 = 30720) beside decodes, as in
"ORCA and chunked prefill", §4-§5; and the shared-prefix decode step of "How
To Scale Your Model notes (7-8)", §3 (six requests sharing 4096 positions plus
1024 private each). Two more shapes (``EXTRA``): speculative decode steps of
k + 1 rows, and a prefill-only ragged batch. Values are fp32 N(0, 1) rounded
to bf16.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    name: str
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    # fixed (q_rows, kv_length) per request, or None when drawn from ``draw``
    requests: Optional[tuple] = None
    # random part: list of (count, q_rows, kv_lo, kv_hi) drawn uniformly;
    # q_rows None means q_rows = kv_length (a whole prompt, S0 = 0)
    draw: Optional[tuple] = None
    # positions shared (same physical pages) by every request; must be a
    # multiple of page_size
    shared_prefix: int = 0
    # pool size in pages (None: exactly the pages used)
    pool_pages: Optional[int] = None
    scale: Optional[float] = None
    seed: int = 0
    description: str = ""


SPECS = {
    "tiny_mixed": WorkloadSpec(
        name="tiny_mixed", n_q_heads=4, n_kv_heads=2, head_dim=64, page_size=16,
        requests=((96, 96), (1, 200), (32, 160)), pool_pages=64, scale=1.0 / 8.0,
        seed=1,
        description="Tiny mixed iteration: A prefill 96/96, B decode 1/200, "
                    "C chunk 32/160; Hq 4 / Hkv 2, D 64, page 16, 64-page pool"),
    "llama2_7b_orca_iteration": WorkloadSpec(
        name="llama2_7b_orca_iteration", n_q_heads=32, n_kv_heads=32, head_dim=128,
        page_size=16, requests=((4096, 4096), (1, 1500), (1, 1700)), seed=2,
        description="Llama-2-7B-shaped layer, one ORCA iteration: A prefill "
                    "4096/4096, B decode 1/1500, C decode 1/1700 (4098 Q rows); "
                    "Hq = Hkv = 32, D 128, page 16"),
    "decode_heavy_gqa4": WorkloadSpec(
        name="decode_heavy_gqa4", n_q_heads=32, n_kv_heads=8, head_dim=128,
        page_size=64, draw=((256, 1, 1024, 8192),), seed=3,
        description="256 decodes q 1, kv ~ U{1024..8192}; Hq 32 / Hkv 8, D 128, "
                    "page 64"),
    "chunked_prefill_mix": WorkloadSpec(
        name="chunked_prefill_mix", n_q_heads=32, n_kv_heads=8, head_dim=128,
        page_size=64, requests=((2048, 32768),), draw=((64, 1, 2048, 32768),),
        seed=4,
        description="chunk 2048 rows at kv 32768 (S0 30720) + 64 decodes "
                    "kv ~ U{2048..32768}; Hq 32 / Hkv 8, D 128, page 64"),
    "shared_prefix_decode": WorkloadSpec(
        name="shared_prefix_decode", n_q_heads=32, n_kv_heads=8, head_dim=128,
        page_size=64, requests=tuple((1, 5121) for _ in range(6)),
        shared_prefix=4096, seed=5,
        description="6 decodes q 1, kv 5121, sharing the physical pages of a "
                    "4096-position prefix + 1025 private positions each; "
                    "Hq 32 / Hkv 8, D 128, page 64"),
    # two further shapes the same triple expresses
    "spec_decode_k3": WorkloadSpec(
        name="spec_decode_k3", n_q_heads=32, n_kv_heads=8, head_dim=128,
        page_size=64, draw=((64, 4, 1024, 8192),), seed=6,
        description="64 speculative-decode steps of k + 1 = 4 rows each (3 draft "
                    "tokens + 1), kv ~ U{1024..8192}; Hq 32 / Hkv 8, D 128, page 64"),
    "varlen_prefill": WorkloadSpec(
        name="varlen_prefill", n_q_heads=32, n_kv_heads=8, head_dim=128,
        page_size=64, draw=((16, None, 128, 4096),), seed=7,
        description="prefill-only varlen batch (cu_seqlens style): 16 requests, "
                    "q_rows = kv ~ U{128..4096}, S0 = 0; Hq 32 / Hkv 8, D 128, page 64"),
}

# The order the pages' workloads are usually listed in.
ORDER = ["tiny_mixed", "llama2_7b_orca_iteration", "decode_heavy_gqa4",
         "chunked_prefill_mix", "shared_prefix_decode"]
# Further shapes: several new rows per decode step (speculative / MTP
# verification, "GLM-5.3 e2e token ledger", stage 3: up to k + 1 tokens per
# running request) and a prefill-only ragged batch ("One forward, many
# requests", §6: cu_seqlens over a flat token buffer).
EXTRA = ["spec_decode_k3", "varlen_prefill"]
ALL = ORDER + EXTRA


@dataclasses.dataclass
class Workload:
    spec: WorkloadSpec
    requests: np.ndarray        # int32 [n, 3]: (q_start, q_end, kv_length)
    block_table: np.ndarray     # int32 [n, max_blocks]; unused entries -1
    num_pages: int
    shared_pages: int           # number of leading pages shared by all requests
    q: torch.Tensor             # bf16 [total_q, Hq, D]
    k_new: torch.Tensor         # bf16 [total_q, Hkv, D]
    v_new: torch.Tensor
    hist_requests: np.ndarray   # int32 [n, 3]: history rows as a prefill of S0 rows
    k_hist: torch.Tensor        # bf16 [sum S0, Hkv, D], logical order per request
    v_hist: torch.Tensor

    @property
    def total_q(self) -> int:
        return int(self.requests[:, 1].max()) if len(self.requests) else 0

    @property
    def n_requests(self) -> int:
        return int(self.requests.shape[0])

    def logical_kv(self, r: int):
        """Logical ``[kv_length, Hkv, D]`` K and V of request ``r`` (history
        followed by this iteration's rows), on the tensors' device."""
        hs, he, _ = self.hist_requests[r]
        qs, qe, _ = self.requests[r]
        k = torch.cat([self.k_hist[hs:he], self.k_new[qs:qe]], 0)
        v = torch.cat([self.v_hist[hs:he], self.v_new[qs:qe]], 0)
        return k, v


def request_shapes(spec: WorkloadSpec) -> list:
    """(q_rows, kv_length) per request, in flat order (fixed part first)."""
    shapes = list(spec.requests or ())
    if spec.draw:
        rng = np.random.default_rng(spec.seed)
        for count, q_rows, lo, hi in spec.draw:
            kvs = rng.integers(lo, hi + 1, size=count)
            shapes += [(int(kv) if q_rows is None else q_rows, int(kv)) for kv in kvs]
    return shapes


def _randn_bf16(shape, gen: torch.Generator, device, chunk_elems=1 << 26):
    """N(0,1) fp32 rounded to bf16, generated in chunks to bound temporaries."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        flat[s:e] = torch.randn(e - s, generator=gen, device=device,
                                dtype=torch.float32).to(torch.bfloat16)
    return out


def make_workload(name_or_spec, device="cpu", seed: Optional[int] = None,
                  with_values: bool = True) -> Workload:
    spec = SPECS[name_or_spec] if isinstance(name_or_spec, str) else name_or_spec
    seed = spec.seed if seed is None else seed
    shapes = request_shapes(spec)
    ps = spec.page_size
    n = len(shapes)

    # flat Q rows and history rows, request by request
    reqs = np.zeros((n, 3), dtype=np.int32)
    hist = np.zeros((n, 3), dtype=np.int32)
    q_off = 0
    h_off = 0
    for r, (q_rows, kv) in enumerate(shapes):
        if q_rows > kv:
            raise ValueError("q_rows > kv_length in workload spec")
        s0 = kv - q_rows
        reqs[r] = (q_off, q_off + q_rows, kv)
        hist[r] = (h_off, h_off + s0, s0)
        q_off += q_rows
        h_off += s0

    # page assignment: a seeded permutation of the pool
    if spec.shared_prefix % ps:
        raise ValueError("shared prefix must be whole pages")
    shared = spec.shared_prefix // ps
    blocks = [math.ceil(kv / ps) for _, kv in shapes]
    private = [b - shared for b in blocks]
    used = shared + sum(private)
    pool = spec.pool_pages or used
    if pool < used:
        raise ValueError("page pool too small")
    rng = np.random.default_rng(seed + 1000)
    perm = rng.permutation(pool).astype(np.int32)
    max_blocks = max(blocks) if blocks else 1
    bt = np.full((n, max_blocks), -1, dtype=np.int32)
    shared_ids = perm[:shared]
    cur = shared
    for r in range(n):
        bt[r, :shared] = shared_ids
        bt[r, shared:blocks[r]] = perm[cur:cur + private[r]]
        cur += private[r]

    hq, hkv, d = spec.n_q_heads, spec.n_kv_heads, spec.head_dim
    if with_values:
        gen = torch.Generator(device=device)
        gen.manual_seed(seed)
        q = _randn_bf16((q_off, hq, d), gen, device)
        k_new = _randn_bf16((q_off, hkv, d), gen, device)
        v_new = _randn_bf16((q_off, hkv, d), gen, device)
        k_hist = _randn_bf16((h_off, hkv, d), gen, device)
        v_hist = _randn_bf16((h_off, hkv, d), gen, device)
        if spec.shared_prefix:
            # the shared positions hold the same K/V for every request: they
            # are one physical copy
            sp = spec.shared_prefix
            h0 = int(hist[0, 0])
            for r in range(1, n):
                hs = int(hist[r, 0])
                k_hist[hs:hs + sp] = k_hist[h0:h0 + sp]
                v_hist[hs:hs + sp] = v_hist[h0:h0 + sp]
    else:
        empty = lambda *s: torch.empty(s, dtype=torch.bfloat16, device=device)  # noqa: E731
        q, k_new, v_new = empty(q_off, hq, d), empty(q_off, hkv, d), empty(q_off, hkv, d)
        k_hist, v_hist = empty(h_off, hkv, d), empty(h_off, hkv, d)

    return Workload(spec=spec, requests=reqs, block_table=bt, num_pages=pool,
                    shared_pages=shared, q=q, k_new=k_new, v_new=v_new,
                    hist_requests=hist, k_hist=k_hist, v_hist=v_hist)
