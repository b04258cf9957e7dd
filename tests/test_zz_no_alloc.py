"""The entry point that allocates nothing (``mb_attn_forward_noalloc``).

Some callers may not allocate device memory (their device memory is owned by
someone else, or a cudaMalloc would stall a hot loop). They plan on the host
only and run the forward with the library's own static scratch array. This
file checks, through the C ABI, that two calls in a row give bit for bit the
results of the regular entry point with a caller-owned workspace (the same
kernels on the same plan), that those results match the fp64 oracle, that a
plan with no rows still reports a clean status word, and that a plan too big
for the array is refused before anything runs. It is collected last so that a
failure here does not hide the other tests' results.
"""

import numpy as np
import pytest
import torch

from continuous_batching_paged_varlen_gb300 import binding as B
from continuous_batching_paged_varlen_gb300 import workloads as W
from tests.gpu_harness import assert_request_close, cfg_of, fill_cache, run_forward

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from continuous_batching_paged_varlen_gb300 import build
    build.build()
    B.lib()


def _bits(t):
    return t.contiguous().view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).cpu()


def _oracle_checks(w, out, lse):
    """Every request against the fp64 oracle; for the 4096-row prefill two
    query heads over its first and last 128 rows."""
    for r in range(w.n_requests):
        m = int(w.requests[r, 1] - w.requests[r, 0])
        if m > 512:
            for rows in ((0, 128), (m - 128, m)):
                assert_request_close(w, out, lse, r, heads=[0, w.spec.n_q_heads - 1], rows=rows)
        else:
            assert_request_close(w, out, lse, r)


@pytest.mark.parametrize("name,opts", [("tiny_mixed", None),
                                       ("shared_prefix_decode", None),
                                       ("llama2_7b_orca_iteration", dict(kv_chunk=256))])
def test_noalloc_matches_workspace_entry_point(name, opts):
    w = W.make_workload(name, device="cuda")
    kc, vc, cfg = fill_cache(w)
    o = B.options(**opts) if opts else None
    ref_out, ref_lse, ref_status, info = run_forward(w, kc, vc, cfg, o)
    assert ref_status == 0
    hp = B.HostPlan(w.requests, w.block_table, cfg, o)
    assert hp.info.workspace_bytes <= 8 << 20
    s = w.spec
    bt = torch.from_numpy(np.ascontiguousarray(w.block_table)).cuda()
    q = w.q.cuda()
    for call in range(2):  # the second call reuses the array the first one left behind
        out = torch.full((w.total_q, s.n_q_heads, s.head_dim), float("nan"),
                         dtype=torch.bfloat16, device="cuda")
        lse = torch.full((w.total_q, s.n_q_heads), float("nan"), device="cuda")
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        B.forward_noalloc(hp, q, kc, vc, bt, out, lse, status)
        torch.cuda.synchronize()
        assert status.item() == 0, f"call {call}: device flags {status.item()}"
        # same plan, same kernels: every output and LSE bit is the same
        assert torch.equal(_bits(out), _bits(ref_out)), f"{name} out, call {call}"
        assert torch.equal(_bits(lse), _bits(ref_lse)), f"{name} lse, call {call}"
        if call == 0:
            _oracle_checks(w, out, lse)
    hp.close()


def test_noalloc_plan_without_rows_clears_the_status_word():
    w = W.make_workload("tiny_mixed")
    reqs = w.requests.copy()
    reqs[:, 1] = reqs[:, 0]  # no request has new rows this iteration
    hp = B.HostPlan(reqs, w.block_table, cfg_of(w))
    assert hp.info.total_q == 0
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    B.forward_noalloc(hp, None, None, None, None, None, None, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    hp.close()


def test_noalloc_rejects_plan_larger_than_the_array():
    w = W.make_workload("decode_heavy_gqa4", with_values=False)
    hp = B.HostPlan(w.requests, w.block_table, cfg_of(w), B.options(kv_chunk=64))
    assert hp.info.workspace_bytes > 8 << 20
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(B.MBError) as e:
        B.forward_noalloc(hp, dummy, dummy, dummy, bt, dummy)
    assert e.value.status == 4  # MB_ERR_WORKSPACE, nothing enqueued
    hp.close()
