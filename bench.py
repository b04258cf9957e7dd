#!/usr/bin/env python
"""Benchmark of one mixed continuous-batching attention step on GB300.

A step is one pass of the whole path over one iteration's synthetic batch:
KV append of the iteration's new rows (``mb_kv_append``), planning with the
one host->device upload of the work lists (``mb_attn_plan``) and the
attention of every request (``mb_attn_forward``: split-KV / cascade kernel
with the LSE merge of split rows inside it, tcgen05 prefill kernel). Inputs
are resident in HBM; between timed steps the L2 is flushed by writing a 256
MiB buffer, then reading another 256 MiB (outside the timed events). Each
step is timed with CUDA events on the launching stream.

Default workload: the Llama-2-7B-shaped layer of one ORCA iteration (a
4096-row prefill beside decodes at kv 1500 and 1700; 32 heads, head dim 128,
page 16). The metric is Q rows per second; the dominant kernel's roofline,
the end-to-end number through host buffers and the CPU oracle's rate on a
bounded sample are reported beside it, one JSON line on stdout.

``--impl reference`` times the fp64 CPU oracle on the host cores instead.
Multi-GPU (torchrun): independent replicas, one per rank, no collective on
the data path; ranks meet only for the barrier and the max-over-ranks time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from continuous_batching_paged_varlen_gb300 import counters as C  # noqa: E402
from continuous_batching_paged_varlen_gb300 import workloads as W  # noqa: E402

METRIC = "mixed-iteration attention Q rows/s; achieved HBM TB/s or tensor-pipe % of peak"
UNIT = "Q rows/s"
DEFAULT_WORKLOAD = "llama2_7b_orca_iteration"
PREFILL_MIN_ROWS = 16  # the planner's default split between the two kernels
FLUSH_BYTES = 256 << 20
SPIN_CYCLES = 1_000_000  # ~0.5 ms of device spin before each per-stage pass
STAGES = ["decode", "prefill"]  # the LSE merge runs inside the split-KV kernels
STAGE_INDEX = {"decode": 0, "prefill": 2}  # MB_STAGE_DECODE, MB_STAGE_PREFILL
KERNEL_SOURCES = {"prefill": "prefill.cu", "decode": "decode.cu", "decode_fp8": "decode_fp8.cu"}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=W.ALL)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="budget of the oracle CPU baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true",
                    help="skip the clock-sampling window (profiling runs)")
    ap.add_argument("--max-requests", type=int, default=0,
                    help="keep only the first N requests of the workload (small profiling "
                         "captures of the same kernels)")
    ap.add_argument("--disable-cascade", action="store_true",
                    help="plan without shared-prefix grouping (comparison runs)")
    ap.add_argument("--rope", action="store_true",
                    help="append through the fused rotary-embedding + KV append "
                         "(mb_rope_kv_append) instead of the plain scatter")
    ap.add_argument("--fp8", action="store_true",
                    help="fp8 (e4m3) KV cache with per-row fp32 scales: quantizing append "
                         "(mb_kv_append_fp8) and mb_attn_forward_fp8 (every request on the "
                         "split-KV path)")
    args = ap.parse_args(argv)
    if args.fp8 and args.rope:
        ap.error("--fp8 and --rope are separate variants")
    return args


def job_throughput(total_ms_local, rows_per_step, steps, world):
    """Whole-job rate of `world` replicas that each timed `steps` steps of
    `rows_per_step` rows: the job takes as long as its slowest rank (max over
    ranks through the default process group when world > 1). Returns (rows/s,
    job milliseconds)."""
    total_ms = float(total_ms_local)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([total_ms], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    return world * rows_per_step * steps / (total_ms / 1e3), total_ms


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, local, world


# --------------------------------------------------------------- peaks

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# --------------------------------------------------------------- algorithmic work

def prefill_request_mask(w, cfg, opts):
    """Which requests the plan runs on the prefill kernel (read from the
    plan's own work list: the planner may also give it short requests)."""
    from continuous_batching_paged_varlen_gb300 import binding as B
    hp = B.HostPlan(w.requests, w.block_table, cfg, opts)
    try:
        n = hp.info.n_prefill_items
        off = hp.layout()[2]
        meta = np.frombuffer(hp.metadata(), dtype=np.uint8)
        recs = np.frombuffer(meta[off:off + 32 * n].tobytes(), dtype=np.int32).reshape(n, 8)
    finally:
        hp.close()
    mask = np.zeros(len(w.requests), dtype=bool)
    mask[np.unique(recs[:, 0])] = True  # field 0: the request (block-table row)
    return mask


def stage_work(w, fp8=False, prefill_mask=None):
    """Algorithmic FLOPs and bytes of the two attention kernels' request sets
    (fp8: every request on the split-KV kernel, 1-byte K/V + fp32 row scales)."""
    s = w.spec
    reqs = w.requests
    m = reqs[:, 1] - reqs[:, 0]
    split_min = (1 << 30) if fp8 else PREFILL_MIN_ROWS
    kvb = dict(kv_elem_bytes=1, kv_row_scale_bytes=4) if fp8 else {}
    on_pre = (m >= split_min) if prefill_mask is None else (prefill_mask & (m > 0))
    pre = reqs[on_pre]
    dec_idx = np.nonzero((m > 0) & ~on_pre)[0]
    dec = reqs[dec_idx]
    out = {}
    out["prefill_flops"] = C.attention_flops(pre, s.n_q_heads, s.head_dim) if len(pre) else 0
    out["prefill_bytes"] = (C.attention_bytes(pre, w.block_table[on_pre],
                                              s.n_q_heads, s.n_kv_heads, s.head_dim,
                                              s.page_size, **kvb) if len(pre) else 0)
    out["decode_flops"] = C.attention_flops(dec, s.n_q_heads, s.head_dim) if len(dec) else 0
    out["decode_bytes"] = (C.attention_bytes(dec, w.block_table[dec_idx], s.n_q_heads,
                                             s.n_kv_heads, s.head_dim, s.page_size, **kvb)
                           if len(dec) else 0)
    out["total_flops"] = C.attention_flops(reqs, s.n_q_heads, s.head_dim)
    out["total_bytes"] = C.attention_bytes(reqs, w.block_table, s.n_q_heads, s.n_kv_heads,
                                           s.head_dim, s.page_size, **kvb)
    out["append_bytes"] = (C.append_fp8_bytes(w.total_q, s.n_kv_heads, s.head_dim) if fp8
                           else C.append_bytes(w.total_q, s.n_kv_heads, s.head_dim))
    return out


def source_hash(kernel):
    path = os.path.join(ROOT, "continuous_batching_paged_varlen_gb300", "csrc",
                        KERNEL_SOURCES[kernel])
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on
    the current source of that kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{kernel}:{workload}")
    if not e or e.get("source_sha256_16") != source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


# --------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names[1:], parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        loaded = [x for x in sm if x > 0.5 * (mx or max(sm))] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- CPU oracle timing

def time_oracle_sample(w, budget_s, rotate=0, fp8=False):
    """Time the fp64 oracle on a bounded sample of workload w; returns
    (Q rows/s extrapolated to the whole workload, description, seconds).
    fp8: each request's K/V go through the oracle's e4m3 quantization and
    dequantization first (timed with the request's first head)."""
    from oracle import attention as OA  # the oracle is only used on this leg
    from oracle import fp8 as OF

    s = w.spec
    g = s.n_q_heads // s.n_kv_heads
    t_total_est = 0.0
    spent = 0.0
    parts = []
    order = sorted(range(w.n_requests), key=lambda r: int(w.requests[r, 1] - w.requests[r, 0]))
    for r in order:
        qs, qe, kv = [int(x) for x in w.requests[r]]
        if qe == qs:
            continue
        k, v = w.logical_kv(r)
        t0 = time.perf_counter()
        if fp8:
            k = OF.dequantize_rows(*OF.quantize_rows(k.to("cpu").float().numpy()))
            v = OF.dequantize_rows(*OF.quantize_rows(v.to("cpu").float().numpy()))
        else:
            k = k.to("cpu").double().numpy()
            v = v.to("cpu").double().numpy()
        q = w.q[qs:qe].to("cpu").double().numpy()
        heads_done = 0
        t_req = (time.perf_counter() - t0) if fp8 else 0.0
        spent += t_req
        for i in range(s.n_q_heads):
            h = (i + rotate) % s.n_q_heads
            kh = h // g
            t0 = time.perf_counter()
            OA.attend(q[:, h:h + 1], k[:, kh:kh + 1], v[:, kh:kh + 1], s.scale)
            dt = time.perf_counter() - t0
            t_req += dt
            heads_done += 1
            spent += dt
            if spent > budget_s:
                break
        t_total_est += t_req * s.n_q_heads / heads_done
        parts.append(f"req{r}(q{qe - qs},kv{kv}):{heads_done}/{s.n_q_heads} heads")
        if spent > budget_s:
            # requests not reached: extrapolate with the per-pair cost seen so far
            done_pairs = sum(C.pairs(int(w.requests[x, 1] - w.requests[x, 0]), int(w.requests[x, 2]))
                             for x in order[:order.index(r) + 1])
            all_pairs = sum(C.pairs(int(a[1] - a[0]), int(a[2])) for a in w.requests)
            if done_pairs < all_pairs:
                t_total_est *= all_pairs / done_pairs
                parts.append(f"rest extrapolated by pairs ({done_pairs}/{all_pairs})")
            break
    rate = w.total_q / t_total_est if t_total_est > 0 else 0.0
    return rate, "; ".join(parts), spent


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# --------------------------------------------------------------- reference arm

def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    w = W.make_workload(args.workload, device="cpu")
    per_step = max(1.0, min(8.0, 150.0 / max(1, args.steps + args.warmup)))
    rates, spents = [], []
    desc = ""
    for i in range(args.warmup + args.steps):
        rate, desc, spent = time_oracle_sample(w, per_step, rotate=i, fp8=args.fp8)
        if i >= args.warmup:
            rates.append(rate)
            spents.append(spent)
    value = statistics.median(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": w.total_q / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config_args(w, args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"per step {statistics.median(spents):.3g} s of fp64 oracle "
                                   f"work (at most ~{per_step:.0f} s): {desc}; rate "
                                   "extrapolated to every head / request"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def truncate(w, n):
    """The first n requests of a workload (same pages, same values)."""
    import dataclasses
    n = min(n, w.n_requests)
    tq = int(w.requests[n - 1, 1])
    th = int(w.hist_requests[n - 1, 1])
    return dataclasses.replace(w, requests=w.requests[:n].copy(),
                               block_table=w.block_table[:n].copy(), q=w.q[:tq],
                               k_new=w.k_new[:tq], v_new=w.v_new[:tq],
                               hist_requests=w.hist_requests[:n].copy(),
                               k_hist=w.k_hist[:th], v_hist=w.v_hist[:th])


def workload_config(w):
    s = w.spec
    return {"workload": s.name, "description": s.description, "q_rows": w.total_q,
            "requests": w.n_requests, "n_q_heads": s.n_q_heads, "n_kv_heads": s.n_kv_heads,
            "head_dim": s.head_dim, "page_size": s.page_size,
            "l2": "flushed between timed steps (256 MiB written, then another 256 MiB read so "
                  "that no dirty line is left to write back; outside the events)",
            "step": "mb_kv_append + mb_attn_plan (host + 1 H2D) + mb_attn_forward",
            "stage_timing": "per-kernel times from a second pass with CUDA events around each "
                            "stage, stages back to back, L2 flushed, a 0.5 ms device spin "
                            "before each pass so the events bracket execution, not host launch "
                            "gaps"}


def workload_config_args(w, args):
    c = workload_config(w)
    if args.max_requests:
        c["max_requests"] = args.max_requests
    if args.disable_cascade:
        c["cascade"] = "disabled"
    if args.rope:
        c["append"] = "fused rotary embedding + KV append (mb_rope_kv_append)"
        c["step"] = "mb_rope_kv_append + mb_attn_plan (host + 1 H2D) + mb_attn_forward"
    if args.fp8:
        c["kv_cache"] = ("fp8 e4m3 codes + one fp32 scale per (token, KV head) row; "
                         "mb_kv_append_fp8 + mb_attn_forward_fp8, every request on the "
                         "split-KV kernel")
        c["step"] = "mb_kv_append_fp8 + mb_attn_plan (host + 1 H2D) + mb_attn_forward_fp8"
    return c


# --------------------------------------------------------------- GPU arm

def run_gpu(args):
    import torch

    from continuous_batching_paged_varlen_gb300 import binding as B
    from continuous_batching_paged_varlen_gb300 import build as build_mod

    rank, local, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build_mod.build()
    B.lib()

    w = W.make_workload(args.workload, device=dev)
    if args.max_requests:
        w = truncate(w, args.max_requests)
    s = w.spec
    opts = None
    if args.disable_cascade or args.fp8:
        opts = B.options(disable_cascade=1 if args.disable_cascade else 0,
                         prefill_min_rows=-1 if args.fp8 else 0)
    cfg = B.config(s.n_q_heads, s.n_kv_heads, s.head_dim, s.page_size, w.num_pages,
                   w.block_table.shape[1], s.scale or 0.0)
    shape = (w.num_pages, s.n_kv_heads, s.page_size, s.head_dim)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if args.fp8:
        kc = torch.zeros(shape, dtype=torch.uint8, device=dev)    # e4m3 codes
        vc = torch.zeros(shape, dtype=torch.uint8, device=dev)
        ksc = torch.zeros(shape[:3], dtype=torch.float32, device=dev)
        vsc = torch.zeros(shape[:3], dtype=torch.float32, device=dev)
    else:
        kc = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
        vc = torch.zeros(shape, dtype=torch.bfloat16, device=dev)

    def append_rows(kn, vn, slot_t):
        if args.fp8:
            B.kv_append_fp8(kc, vc, ksc, vsc, kn, vn, slot_t, cfg, status)
        else:
            B.kv_append(kc, vc, kn, vn, slot_t, cfg, status)

    def forward(plan, q_t, events=None, o=None, l=None):
        o = out if o is None else o
        l = lse if l is None else l
        if args.fp8:
            plan.forward_fp8(q_t, kc, vc, ksc, vsc, bt_dev, o, l, events=events)
        else:
            plan.forward(q_t, kc, vc, bt_dev, o, l, events=events)

    n_hist = int(w.hist_requests[:, 1].max()) if w.n_requests else 0
    if n_hist:
        hs = B.slot_mapping(w.hist_requests, w.block_table, cfg, n_hist)
        append_rows(w.k_hist, w.v_hist, torch.from_numpy(hs).to(dev))
    slots = torch.from_numpy(B.slot_mapping(w.requests, w.block_table, cfg, w.total_q)).to(dev)
    if args.rope:
        pos_dev = torch.from_numpy(B.positions(w.requests, w.total_q)).to(dev)
        rope_tab = torch.from_numpy(
            B.rope_table(int(w.requests[:, 2].max()) + 1, s.head_dim)).to(dev)
        q_rot = w.q.clone()  # rotated in place every step (timing only)
    bt_dev = torch.from_numpy(np.ascontiguousarray(w.block_table)).to(dev)
    q, k_new, v_new = w.q, w.k_new, w.v_new
    out = torch.empty((w.total_q, s.n_q_heads, s.head_dim), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.total_q, s.n_q_heads), dtype=torch.float32, device=dev)
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    class _Flush:
        """Cold L2 before a timed region: writing 256 MiB evicts every line
        the step could reuse; reading another 256 MiB then evicts (writes
        back) those dirty lines, so the next step does not pay for the
        flush's own write-back."""

        @staticmethod
        def zero_():
            flush_w.zero_()
            flush_r.max()

    flush = _Flush()
    stream = torch.cuda.current_stream(dev)
    probe = B.Plan(w.requests, w.block_table, cfg, device=dev, opts=opts)
    info = probe.info.as_dict()
    ws = probe.workspace
    probe.close()
    launches_per_step = 1 + info["n_launches"]

    def append():
        if args.rope:
            B.rope_kv_append(q_rot, kc, vc, k_new, v_new, pos_dev, slots, rope_tab, cfg, status)
        else:
            append_rows(k_new, v_new, slots)

    def step(stage_events=None):
        append()
        plan = B.Plan(w.requests, w.block_table, cfg, device=dev, workspace=ws, opts=opts)
        forward(plan, q, stage_events)
        plan.close()

    def kernel_pass(stage_events, append_events):
        # the same launches with per-stage events (stages back to back). A
        # device spin first (torch's, about half a millisecond) lets the host
        # enqueue the whole pass before the GPU reaches it, so each event pair
        # brackets its kernel's execution, not the host's launch work.
        torch.cuda._sleep(SPIN_CYCLES)
        append_events[0].record(stream)
        append()
        append_events[1].record(stream)
        plan = B.Plan(w.requests, w.block_table, cfg, device=dev, workspace=ws, opts=opts)
        forward(plan, q, stage_events)
        plan.close()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * B.NUM_STAGES)]
           for _ in range(K)]
    aev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    for row in sev:  # torch creates the CUDA event on first record: do it here so the
        for e in row:  # library receives real handles
            e.record(stream)
    clocks = ClockSampler(local)
    # nvidia-smi samples every 200 ms: the timed region is embedded in a
    # window of identical untimed steps (>= 1 s before, >= 0.3 s after) so the
    # samples show the clocks the timed steps ran at
    if not args.no_clocks:
        clocks.start()
    t_end = time.perf_counter() + (0.0 if args.no_clocks else 1.0)
    while time.perf_counter() < t_end:
        flush.zero_()
        step()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    host_s = 0.0
    for i in range(K):
        flush.zero_()
        ev[i][0].record(stream)
        h0 = time.perf_counter()
        step()
        host_s += time.perf_counter() - h0
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    t_end = time.perf_counter() + (0.0 if args.no_clocks else 0.3)
    while time.perf_counter() < t_end:
        flush.zero_()
        step()
        torch.cuda.synchronize()
    clk = clocks.stop()
    # per-kernel durations for the roofline: the same launches again, each
    # stage bracketed by its own events (L2 flushed before every pass)
    for i in range(K):
        flush.zero_()
        kernel_pass(sev[i], aev[i])
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    stage_ms = {}
    for name in STAGES:
        si = STAGE_INDEX[name]
        if info[{"decode": "n_decode_items", "prefill": "n_prefill_items"}[name]] > 0:
            stage_ms[name] = statistics.mean(
                sev[i][2 * si].elapsed_time(sev[i][2 * si + 1]) for i in range(K))
    stage_ms["append"] = statistics.mean(a.elapsed_time(b) for a, b in aev)
    ms_step = statistics.mean(step_ms)
    value, total_ms = job_throughput(sum(step_ms), w.total_q, K, world)
    dev_status = int(ws[:4].view(torch.int32).item()) | int(status.item())

    # ---- roofline of the dominant kernel
    peaks = load_peaks()
    work = stage_work(w, fp8=args.fp8, prefill_mask=prefill_request_mask(w, cfg, opts))
    if args.rope:
        work["append_bytes"] = C.rope_append_bytes(w.total_q, s.n_q_heads, s.n_kv_heads,
                                                   s.head_dim)
    dominant = max(stage_ms, key=stage_ms.get) if stage_ms else None
    roof = None
    if dominant == "prefill":
        t = stage_ms["prefill"] / 1e3
        ach = work["prefill_flops"] / t / 1e12
        roof = {"kernel": "prefill_kernel (tcgen05)", "bound": "tensor", "achieved": ach,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / peaks["bf16_tflops"],
                "peak_kind": f"bf16 dense burst ({peaks['source']})",
                "algorithmic_per_launch": work["prefill_flops"],
                "traffic": recorded_traffic("prefill", s.name)}
    elif dominant == "append":
        t = stage_ms["append"] / 1e3
        ach = work["append_bytes"] / t / 1e9
        roof = {"kernel": ("rope_append_kernel" if args.rope else
                           "kv_append_fp8_kernel" if args.fp8 else "kv_append_kernel"),
                "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "peak_kind": f"HBM copy ({peaks['source']})",
                "algorithmic_per_launch": work["append_bytes"], "traffic": None}
    elif dominant == "decode":
        t = stage_ms["decode"] / 1e3
        ach = work["decode_bytes"] / t / 1e9
        roof = {"kernel": "splitkv_fp8_kernel" if args.fp8 else "splitkv_kernel",
                "bound": "hbm", "achieved": ach,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
                "peak_kind": f"HBM copy ({peaks['source']})",
                "algorithmic_per_launch": work["decode_bytes"],
                "traffic": recorded_traffic("decode_fp8" if args.fp8 else "decode", s.name)}

    # ---- end to end through host buffers
    e2e = None
    if not args.no_e2e:
        hq = q.cpu().pin_memory()
        hk = k_new.cpu().pin_memory()
        hv = v_new.cpu().pin_memory()
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k_new), torch.empty_like(v_new)

        def e2e_step():
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            append_rows(dk, dv, slots)
            plan = B.Plan(w.requests, w.block_table, cfg, device=dev, workspace=ws, opts=opts)
            forward(plan, dq)
            plan.close()
            hout.copy_(out, non_blocking=True)
            hlse.copy_(lse, non_blocking=True)

        for _ in range(max(3, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        e_ms = []
        for i in range(K):
            flush.zero_()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            e2e_step()
            torch.cuda.synchronize()
            e_ms.append((time.perf_counter() - t0) * 1e3)

        # A serving loop keeps steps in flight: step i's upload (its own
        # stream) overlaps step i-1's attention, and its download (a third
        # stream) overlaps step i+1's upload. Inputs, outputs and plan
        # workspaces rotate over NBUF buffer sets; every step still plans,
        # uploads its Q/K/V and downloads its O/LSE. The plan is made on the
        # upload stream, ahead of the step's inputs: its work-list copy then
        # shares the copy engine's queue in order, instead of waiting on the
        # compute stream behind the next step's 100 MB upload.
        NBUF = 3
        s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        bufs = [dict(q=torch.empty_like(q), k=torch.empty_like(k_new), v=torch.empty_like(v_new),
                     o=torch.empty_like(out), l=torch.empty_like(lse), ws=torch.empty_like(ws),
                     ho=torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                     hl=torch.empty(lse.shape, dtype=lse.dtype).pin_memory(),
                     free=torch.cuda.Event(), up=torch.cuda.Event(), done=torch.cuda.Event())
                for _ in range(NBUF)]

        def piped_step(i):
            b = bufs[i % NBUF]
            with torch.cuda.stream(s_up):
                if i >= NBUF:  # step i-NBUF has been computed and downloaded
                    s_up.wait_event(b["free"])
                plan = B.Plan(w.requests, w.block_table, cfg, device=dev, workspace=b["ws"],
                              opts=opts, stream=s_up)
                b["q"].copy_(hq, non_blocking=True)
                b["k"].copy_(hk, non_blocking=True)
                b["v"].copy_(hv, non_blocking=True)
                b["up"].record(s_up)
            stream.wait_event(b["up"])
            append_rows(b["k"], b["v"], slots)
            forward(plan, b["q"], o=b["o"], l=b["l"])
            plan.close()
            b["done"].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(b["done"])
                b["ho"].copy_(b["o"], non_blocking=True)
                b["hl"].copy_(b["l"], non_blocking=True)
                b["free"].record(s_down)

        for i in range(max(3, args.warmup)):
            piped_step(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(K):
            piped_step(i)
        torch.cuda.synchronize()
        piped_ms = (time.perf_counter() - t0) * 1e3 / K
        h2d = (hq.numel() + hk.numel() + hv.numel()) * 2 + info["metadata_bytes"]
        d2h = hout.numel() * 2 + hlse.numel() * 4
        e2e = {"value": world * w.total_q / (piped_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": piped_ms,
               "timing": "K steps through the public calls, pipelined (each step's Q/K/V "
                         "upload from pinned host memory and its plan on an upload stream, "
                         "append + forward on the compute stream, O/LSE download on a third "
                         "stream; inputs, outputs and workspaces rotate over 3 buffer sets); "
                         "host wall clock over "
                         "the K steps, synchronised at both ends",
               "serial": {"value": world * w.total_q / (statistics.mean(e_ms) / 1e3),
                          "ms_per_step": statistics.mean(e_ms),
                          "timing": "one step at a time: host wall clock around each step, "
                                    "synchronised, L2 flushed before it"}}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, desc, spent = time_oracle_sample(w, args.cpu_seconds, fp8=args.fp8)
        cpu = {"value": rate, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{spent:.1f} s of fp64 oracle work: {desc}; extrapolated to every "
                         "head / request of the workload"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 KV + bf16" if args.fp8 else "bf16", "data": "synthetic",
        "config": {**workload_config_args(w, args), "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
        "stages_ms": stage_ms,
        "achieved": {"attention_tflops": work["total_flops"] / (ms_step / 1e3) / 1e12,
                     "attention_hbm_gbs": work["total_bytes"] / (ms_step / 1e3) / 1e9,
                     "algorithmic_flops_per_step": work["total_flops"],
                     "algorithmic_bytes_per_step": work["total_bytes"] + work["append_bytes"],
                     "append_hbm_gbs": work["append_bytes"] / (stage_ms["append"] / 1e3) / 1e9},
        "plan": info, "device_status": dev_status, "wall_s_timed_region": wall,
        # host time to enqueue one step (append, plan + upload, forward, through
        # the Python binding); a step shorter than this on the device is
        # host-bound, the GPU waiting for its launches
        "host_enqueue_us_per_step": host_s / K * 1e6,
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0 if dev_status == 0 else 3


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
