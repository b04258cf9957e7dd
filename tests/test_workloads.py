"""Seeded workload shapes and the bench's counters (no GPU)."""

import json
import os

import numpy as np
import pytest
import torch

from continuous_batching_paged_varlen_gb300 import counters as C
from continuous_batching_paged_varlen_gb300 import workloads as W
from tests.conftest import GOLDEN


def golden_figures():
    with open(os.path.join(GOLDEN, "analytic_figures.json")) as f:
        return json.load(f)


def test_counters_reproduce_printed_figures():
    g = golden_figures()
    x = g["kv_bytes_per_position"]
    assert C.bytes_per_position(**x["inputs"]) == x["value"] == 128 * 1024
    x = g["flops_per_pair_network"]
    assert C.flops_per_pair(x["inputs"]["head_dim"], x["inputs"]["n_heads"],
                            x["inputs"]["n_layers"]) == x["value"]
    assert abs(x["value"] / 1e6 - 0.52) < 0.01
    # causal prefill of length L: L(L+1)/2 pairs ~ L^2/2 -> 2.6e5 * L^2 FLOPs
    L = 4096
    coeff = C.pairs(L, L) * C.flops_per_pair(128, 32, 32) / L ** 2
    assert abs(coeff - g["causal_prefill_flops_coefficient"]["value"]) / 2.6e5 < 0.02
    # shared prefix: 3.75 GiB naive vs 1.25 GiB stored over 32 layers
    per_pos = C.bytes_per_position(32, 8, 128)
    inp = g["shared_prefix_naive_read_gib"]["inputs"]
    n, sp, pp = inp["requests"], inp["shared_positions"], inp["private_positions"]
    reqs = np.array([(r, r + 1, sp + pp) for r in range(n)])
    ps = 64
    bt = np.zeros((n, (sp + pp) // ps), dtype=np.int64)
    for r in range(n):
        bt[r, :sp // ps] = np.arange(sp // ps)
        bt[r, sp // ps:] = sp // ps + r * (pp // ps) + np.arange(pp // ps)
    naive = C.naive_kv_positions(reqs) * per_pos / 2 ** 30
    stored = C.distinct_kv_positions(reqs, bt, ps) * per_pos / 2 ** 30
    assert naive == pytest.approx(g["shared_prefix_naive_read_gib"]["value"])
    assert stored == pytest.approx(g["shared_prefix_stored_gib"]["value"])


def test_tiny_mixed_shape():
    w = W.make_workload("tiny_mixed")
    assert w.requests.tolist() == [[0, 96, 96], [96, 97, 200], [97, 129, 160]]
    assert w.num_pages == 64
    used = w.block_table[w.block_table >= 0]
    assert len(used) == 6 + 13 + 10 == 29 and len(set(used.tolist())) == 29
    assert used.max() < 64
    assert w.q.shape == (129, 4, 64) and w.q.dtype == torch.bfloat16
    assert w.k_new.shape == (129, 2, 64)
    assert w.k_hist.shape == (0 + 199 + 128, 2, 64)
    assert w.hist_requests.tolist() == [[0, 0, 0], [0, 199, 199], [199, 327, 128]]


def test_llama_iteration_shape_and_counts():
    w = W.make_workload("llama2_7b_orca_iteration", with_values=False)
    assert w.total_q == 4098
    assert w.num_pages == 256 + 94 + 107 == 457
    flops = C.attention_flops(w.requests, 32, 128)
    # 4096 * 4097 / 2 causal pairs + 1500 + 1700 decode pairs, 32 heads, D 128
    assert flops == (4096 * 4097 // 2 + 1500 + 1700) * 4 * 128 * 32
    assert abs(flops / 1e9 - 137.9) < 0.5


def test_decode_heavy_shape():
    w = W.make_workload("decode_heavy_gqa4", with_values=False)
    kv = w.requests[:, 2]
    assert len(kv) == 256 and kv.min() >= 1024 and kv.max() <= 8192
    assert (w.requests[:, 1] - w.requests[:, 0] == 1).all()
    assert w.num_pages == int(np.ceil(kv / 64).sum())
    # same seed -> same draw
    w2 = W.make_workload("decode_heavy_gqa4", with_values=False)
    assert np.array_equal(w.block_table, w2.block_table)


def test_chunked_mix_shape():
    w = W.make_workload("chunked_prefill_mix", with_values=False)
    assert w.requests[0].tolist() == [0, 2048, 32768]
    assert len(w.requests) == 65
    kv = w.requests[1:, 2]
    assert kv.min() >= 2048 and kv.max() <= 32768


def test_shared_prefix_shape():
    w = W.make_workload("shared_prefix_decode")
    assert w.shared_pages == 64
    for r in range(6):
        assert np.array_equal(w.block_table[r, :64], w.block_table[0, :64])
        assert (w.block_table[r, 64:81] >= 0).all()
    priv = w.block_table[:, 64:81].ravel()
    assert len(set(priv.tolist())) == 6 * 17
    assert w.num_pages == 64 + 6 * 17
    # identical K/V for the shared positions (one physical copy)
    for r in range(1, 6):
        k0, v0 = w.logical_kv(0)
        kr, vr = w.logical_kv(r)
        assert torch.equal(k0[:4096], kr[:4096]) and torch.equal(v0[:4096], vr[:4096])
    # per layer: 120 MiB naive vs 40 MiB distinct (+ new rows)
    per_pos = 2 * 8 * 128 * 2
    naive = C.naive_kv_positions(w.requests) * per_pos / 2 ** 20
    distinct = C.distinct_kv_positions(w.requests, w.block_table, 64) * per_pos / 2 ** 20
    assert naive == pytest.approx(120.02, abs=0.01)
    assert distinct == pytest.approx(40.02, abs=0.01)


def test_values_are_seeded_bf16_normal():
    a = W.make_workload("tiny_mixed")
    b = W.make_workload("tiny_mixed")
    assert torch.equal(a.q, b.q) and torch.equal(a.k_hist, b.k_hist)
    c = W.make_workload("tiny_mixed", seed=99)
    assert not torch.equal(a.q, c.q)
    x = a.q.float()
    assert abs(x.mean().item()) < 0.05 and abs(x.std().item() - 1.0) < 0.05
