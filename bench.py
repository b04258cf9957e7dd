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
bounded sample are reported beside it, one JSON line on stdout. The default
line also carries ``workloads``: the decode-heavy batch, the chunked-prefill
mix and the shared-prefix step, each timed with the same protocol.

``--impl reference`` times the fp64 CPU oracle on the host cores instead.
Multi-GPU (torchrun): independent replicas, one per rank, no collective on
the data path; ranks meet only for the barrier and the max-over-ranks time.
"""

from __future__ import annotations

import argparse
import contextlib
import ctypes
import hashlib
import json
import os
import re
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
# further workloads of the default line: the decode-dominated batch, the
# chunked-prefill iteration and the shared-prefix decode step
LINE_WORKLOADS = ["decode_heavy_gqa4", "chunked_prefill_mix", "shared_prefix_decode"]
PREFILL_MIN_ROWS = 16  # the planner's default split between the two kernels
FLUSH_BYTES = 256 << 20
SPIN_CYCLES = 1_000_000  # ~0.5 ms of device spin before each per-stage pass
STAGES = ["decode", "prefill"]  # the LSE merge runs inside the split-KV kernels
STAGE_INDEX = {"decode": 0, "prefill": 2}  # MB_STAGE_DECODE, MB_STAGE_PREFILL
CSRC = os.path.join(ROOT, "continuous_batching_paged_varlen_gb300", "csrc")
KERNEL_SOURCES = {"prefill": "prefill.cu", "decode": "decode.cu", "decode_fp8": "decode_fp8.cu"}
MAX_LAYER_CACHE_BYTES = 64 << 30  # --layers: per-layer caches must fit this


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=W.ALL)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="budget of the oracle CPU baseline sample (all cores; the "
                         "one-thread sample gets half of it)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time the chosen workload only (no 'workloads' object)")
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
                         "(mb_kv_append_fp8) and mb_attn_forward_fp8")
    ap.add_argument("--prefill-ctas", type=int, default=0,
                    help="planner option: SMs of the prefill grid beside the split-KV kernel "
                         "(0: the planner's model, < 0: every SM)")
    ap.add_argument("--kv-chunk", type=int, default=0,
                    help="planner option: split-KV chunk in keys (multiple of 64; 0: the "
                         "planner's choice)")
    ap.add_argument("--layers", type=int, default=1,
                    help="a step runs this many layers, each with its own cache: one plan, "
                         "then append + forward per layer, back to back")
    args = ap.parse_args(argv)
    if args.fp8 and args.rope:
        ap.error("--fp8 and --rope are separate variants")
    if args.layers < 1:
        ap.error("--layers must be >= 1")
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
    (fp8: 1-byte K/V + fp32 row scales)."""
    s = w.spec
    reqs = w.requests
    m = reqs[:, 1] - reqs[:, 0]
    kvb = dict(kv_elem_bytes=1, kv_row_scale_bytes=4) if fp8 else {}
    on_pre = (m >= PREFILL_MIN_ROWS) if prefill_mask is None else (prefill_mask & (m > 0))
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


_INCLUDE = re.compile(r'^\s*#\s*include\s+"([^"]+)"', re.M)


def compiled_files(src):
    """The source file and every local header it includes, transitively."""
    seen, todo = [], [os.path.normpath(os.path.join(CSRC, src))]
    while todo:
        p = todo.pop()
        if p in seen or not os.path.exists(p):
            continue
        seen.append(p)
        with open(p) as f:
            for inc in _INCLUDE.findall(f.read()):
                todo.append(os.path.normpath(os.path.join(os.path.dirname(p), inc)))
    return sorted(seen)


def source_hash(kernel):
    """sha256[:16] over the kernel's translation unit: its .cu file and every
    local header it compiles (path relative to the repository + contents)."""
    h = hashlib.sha256()
    for p in compiled_files(KERNEL_SOURCES[kernel]):
        h.update(os.path.relpath(p, ROOT).encode() + b"\0")
        with open(p, "rb") as f:
            h.update(f.read())
        h.update(b"\0")
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on
    the current sources of that kernel (else None)."""
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

class BlasThreads:
    """Thread count of numpy's OpenBLAS, through its own C entry points (found
    among the libraries this process has loaded); ``None`` where none is
    found (then the library's default stands and is reported as unknown)."""

    NAMES = [("scipy_openblas_set_num_threads64_", "scipy_openblas_get_num_threads64_"),
             ("scipy_openblas_set_num_threads", "scipy_openblas_get_num_threads"),
             ("openblas_set_num_threads64_", "openblas_get_num_threads64_"),
             ("openblas_set_num_threads", "openblas_get_num_threads")]

    def __init__(self):
        self.set_fn = self.get_fn = None
        np.dot(np.ones((64, 64)), np.ones((64, 64)))  # make sure BLAS is loaded
        paths = set()
        try:
            with open("/proc/self/maps") as f:
                for line in f:
                    p = line.split()[-1] if line.split() else ""
                    if "blas" in os.path.basename(p).lower() and ".so" in p:
                        paths.add(p)
        except OSError:
            return
        for p in sorted(paths):
            try:
                lib = ctypes.CDLL(p)
            except OSError:
                continue
            for s, g in self.NAMES:
                if hasattr(lib, s) and hasattr(lib, g):
                    self.set_fn, self.get_fn = getattr(lib, s), getattr(lib, g)
                    self.get_fn.restype = ctypes.c_int
                    self.set_fn.argtypes = [ctypes.c_int]
                    return

    def get(self):
        return int(self.get_fn()) if self.get_fn else None

    @contextlib.contextmanager
    def threads(self, n):
        old = self.get()
        if self.set_fn:
            self.set_fn(int(n))
        try:
            yield self.get()
        finally:
            if self.set_fn and old:
                self.set_fn(old)


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


def cpu_baseline(w, budget_s, fp8=False):
    """The oracle timed twice on a bounded sample: BLAS on every core this
    process may run on, then on one thread (half the budget)."""
    blas = BlasThreads()
    cores = cpu_cores()
    with blas.threads(cores) as used:
        rate, desc, spent = time_oracle_sample(w, budget_s, fp8=fp8)
    with blas.threads(1) as used1:
        rate1, desc1, spent1 = time_oracle_sample(w, budget_s / 2, fp8=fp8)
    return {"value": rate, "unit": UNIT, "cores": used if used else cores, "kind": "oracle",
            "blas_threads": used, "affinity_cores": cores,
            "sample": f"{spent:.1f} s of fp64 oracle work with {used or 'default'} BLAS "
                      f"threads: {desc}; extrapolated to every head / request of the workload",
            "one_thread": {"value": rate1, "blas_threads": used1,
                           "sample": f"{spent1:.1f} s: {desc1}"}}


# --------------------------------------------------------------- reference arm

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


def workload_config_args(w, args, world=1):
    """The line's ``config``; the same for both arms of one invocation."""
    c = workload_config(w)
    if args.max_requests:
        c["max_requests"] = args.max_requests
    if args.disable_cascade:
        c["cascade"] = "disabled"
    if args.prefill_ctas:
        c["prefill_ctas"] = args.prefill_ctas
    if args.kv_chunk:
        c["kv_chunk"] = args.kv_chunk
    if args.rope:
        c["append"] = "fused rotary embedding + KV append (mb_rope_kv_append)"
        c["step"] = "mb_rope_kv_append + mb_attn_plan (host + 1 H2D) + mb_attn_forward"
    if args.fp8:
        c["kv_cache"] = ("fp8 e4m3 codes + one fp32 scale per (token, KV head) row; "
                         "mb_kv_append_fp8 + mb_attn_forward_fp8 (prefill requests: their "
                         "pages dequantized to bf16 staging, then the tensor-core kernel)")
        c["step"] = "mb_kv_append_fp8 + mb_attn_plan (host + 1 H2D) + mb_attn_forward_fp8"
    if args.layers > 1:
        c["layers"] = args.layers
        c["step"] = (f"mb_attn_plan once, then {args.layers} x (append + forward), one KV "
                     "cache per layer")
    c["parallelism"] = f"replicas x{world}" if world > 1 else "1 GPU"
    return c


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    w = W.make_workload(args.workload, device="cpu")
    per_step = max(1.0, min(8.0, 150.0 / max(1, args.steps + args.warmup)))
    rates, spents = [], []
    desc = ""
    blas = BlasThreads()
    with blas.threads(cpu_cores()) as used:
        for i in range(args.warmup + args.steps):
            rate, desc, spent = time_oracle_sample(w, per_step, rotate=i, fp8=args.fp8)
            if i >= args.warmup:
                rates.append(rate)
                spents.append(spent)
    # a step of the GPU arm runs every layer: the oracle's per-layer rate / layers
    value = statistics.median(rates) / args.layers
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": w.total_q / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config_args(w, args, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used or cpu_cores(),
                         "kind": "oracle", "blas_threads": used,
                         "sample": f"per step {statistics.median(spents):.3g} s of fp64 oracle "
                                   f"work (at most ~{per_step:.0f} s) with {used or 'default'} "
                                   f"BLAS threads: {desc}; rate extrapolated to every head / "
                                   "request" + (f" and {args.layers} layers" if args.layers > 1
                                                else "")},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def truncate(w, n):
    """The first n requests of a workload, same values, with the page pool
    cut down to the pages they use (renumbered in the same relative order),
    so that a small profiling case holds little device memory."""
    import dataclasses
    n = min(n, w.n_requests)
    tq = int(w.requests[n - 1, 1])
    th = int(w.hist_requests[n - 1, 1])
    bt = w.block_table[:n]
    used = np.unique(bt[bt >= 0])
    remap = np.full(w.num_pages, -1, dtype=np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    bt = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
    return dataclasses.replace(w, requests=w.requests[:n].copy(), block_table=bt,
                               num_pages=int(len(used)), q=w.q[:tq].clone(),
                               k_new=w.k_new[:tq].clone(), v_new=w.v_new[:tq].clone(),
                               hist_requests=w.hist_requests[:n].copy(),
                               k_hist=w.k_hist[:th].clone(), v_hist=w.v_hist[:th].clone())


# --------------------------------------------------------------- GPU arm

def roofline(dominant, stage_ms, work, peaks, kernel_names, workload, fp8):
    """The dominant kernel's achieved rate against its roofline."""
    if dominant == "prefill":
        t = stage_ms["prefill"] / 1e3
        ach = work["prefill_flops"] / t / 1e12
        return {"kernel": kernel_names["prefill"], "bound": "tensor", "achieved": ach,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / peaks["bf16_tflops"],
                "peak_kind": f"bf16 dense burst ({peaks['source']})",
                "algorithmic_per_launch": work["prefill_flops"],
                "traffic": recorded_traffic("prefill", workload) if not fp8 else None}
    if dominant == "append":
        t = stage_ms["append"] / 1e3
        ach = work["append_bytes"] / t / 1e9
        return {"kernel": kernel_names["append"], "bound": "hbm", "achieved": ach,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
                "peak_kind": f"HBM copy ({peaks['source']})",
                "algorithmic_per_launch": work["append_bytes"], "traffic": None}
    if dominant == "decode":
        t = stage_ms["decode"] / 1e3
        ach = work["decode_bytes"] / t / 1e9
        return {"kernel": kernel_names["decode"], "bound": "hbm", "achieved": ach,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
                "peak_kind": f"HBM copy ({peaks['source']})",
                "algorithmic_per_launch": work["decode_bytes"],
                "traffic": recorded_traffic("decode_fp8" if fp8 else "decode", workload)}
    return None


def combined_bound(work, ms_step, peaks, layers=1):
    """max(bytes / HBM, FLOPs / tensor peak) of the whole step against its
    time: the step's own roofline, both halves of a mixed iteration at once."""
    b = layers * (work["total_bytes"] + work["append_bytes"])
    f = layers * work["total_flops"]
    b_ms = b / (peaks["hbm_gbs"] * 1e9) * 1e3
    f_ms = f / (peaks["bf16_tflops"] * 1e12) * 1e3
    return {"bytes": int(b), "flops": int(f), "bytes_ms": b_ms, "flops_ms": f_ms,
            "bound_ms": max(b_ms, f_ms), "frac": max(b_ms, f_ms) / ms_step,
            "hbm_frac": b_ms / ms_step, "tensor_frac": f_ms / ms_step,
            "peaks": f"HBM {peaks['hbm_gbs']} GB/s, bf16 {peaks['bf16_tflops']} TFLOP/s "
                     f"({peaks['source']})"}


def measure(args, name, dev, local, world, *, main):
    """Time one workload (steps, then a per-stage pass); main: also the
    end-to-end number and the workload tensors for the CPU baseline."""
    import torch

    from continuous_batching_paged_varlen_gb300 import binding as B

    L = args.layers if main else 1
    fp8, rope = (args.fp8, args.rope) if main else (False, False)
    w = W.make_workload(name, device=dev)
    if main and args.max_requests:
        w = truncate(w, args.max_requests)
        torch.cuda.empty_cache()
    s = w.spec
    opts = None
    if main and (args.disable_cascade or args.prefill_ctas or args.kv_chunk or fp8):
        opts = B.options(disable_cascade=1 if args.disable_cascade else 0,
                         prefill_ctas=args.prefill_ctas, kv_chunk=args.kv_chunk,
                         fp8_cache=1 if fp8 else 0)
    cfg = B.config(s.n_q_heads, s.n_kv_heads, s.head_dim, s.page_size, w.num_pages,
                   w.block_table.shape[1], s.scale or 0.0)
    shape = (w.num_pages, s.n_kv_heads, s.page_size, s.head_dim)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    n_slots = int(np.prod(shape[:3]))  # (page, KV head, slot) rows of one cache
    per_layer = 2 * n_slots * (s.head_dim + 4 if fp8 else 2 * s.head_dim)  # K and V bytes
    if L > 1 and per_layer * L > MAX_LAYER_CACHE_BYTES:
        raise SystemExit(f"--layers {L}: {per_layer * L / 2**30:.1f} GiB of caches is too much")
    if fp8:
        caches = [(torch.zeros(shape, dtype=torch.uint8, device=dev),
                   torch.zeros(shape, dtype=torch.uint8, device=dev),
                   torch.zeros(shape[:3], dtype=torch.float32, device=dev),
                   torch.zeros(shape[:3], dtype=torch.float32, device=dev))]
    else:
        caches = [(torch.zeros(shape, dtype=torch.bfloat16, device=dev),
                   torch.zeros(shape, dtype=torch.bfloat16, device=dev))]

    def append_rows(c, kn, vn, slot_t):
        if fp8:
            B.kv_append_fp8(c[0], c[1], c[2], c[3], kn, vn, slot_t, cfg, status)
        else:
            B.kv_append(c[0], c[1], kn, vn, slot_t, cfg, status)

    bt_dev = torch.from_numpy(np.ascontiguousarray(w.block_table)).to(dev)
    out = torch.empty((w.total_q, s.n_q_heads, s.head_dim), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.total_q, s.n_q_heads), dtype=torch.float32, device=dev)

    def forward(plan, c, q_t, events=None, o=None, l=None):
        o = out if o is None else o
        l = lse if l is None else l
        if fp8:
            plan.forward_fp8(q_t, c[0], c[1], c[2], c[3], bt_dev, o, l, events=events)
        else:
            plan.forward(q_t, c[0], c[1], bt_dev, o, l, events=events)

    n_hist = int(w.hist_requests[:, 1].max()) if w.n_requests else 0
    if n_hist:
        hs = B.slot_mapping(w.hist_requests, w.block_table, cfg, n_hist)
        append_rows(caches[0], w.k_hist, w.v_hist, torch.from_numpy(hs).to(dev))
    for _ in range(1, L):  # every layer holds the same history (timing only)
        caches.append(tuple(t.clone() for t in caches[0]))
    # the history tensors are not needed on the device any more (the CPU
    # baseline of the main workload reads them back, so those stay)
    slots = torch.from_numpy(B.slot_mapping(w.requests, w.block_table, cfg, w.total_q)).to(dev)
    if rope:
        pos_dev = torch.from_numpy(B.positions(w.requests, w.total_q)).to(dev)
        rope_tab = torch.from_numpy(
            B.rope_table(int(w.requests[:, 2].max()) + 1, s.head_dim)).to(dev)
        q_rot = w.q.clone()  # rotated in place every step (timing only)
    q, k_new, v_new = w.q, w.k_new, w.v_new
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def flush():
        """Cold L2 before a timed region: writing 256 MiB evicts every line
        the step could reuse; reading another 256 MiB then evicts (writes
        back) those dirty lines, so the next step does not pay for the
        flush's own write-back."""
        flush_w.zero_()
        flush_r.max()

    stream = torch.cuda.current_stream(dev)
    probe = B.Plan(w.requests, w.block_table, cfg, device=dev, opts=opts)
    info = probe.info.as_dict()
    ws = probe.workspace
    probe.close()
    launches_per_step = L * (1 + info["n_launches"])

    def append(c):
        if rope:
            B.rope_kv_append(q_rot, c[0], c[1], k_new, v_new, pos_dev, slots, rope_tab, cfg,
                             status)
        else:
            append_rows(c, k_new, v_new, slots)

    def step():
        # returns the host time of mb_attn_plan (planning and the one upload
        # enqueued), which the line reports on its own
        t0 = time.perf_counter()
        plan = B.Plan(w.requests, w.block_table, cfg, device=dev, workspace=ws, opts=opts)
        t_plan = time.perf_counter() - t0
        for c in caches:
            append(c)
            forward(plan, c, q)
        plan.close()
        return t_plan

    def kernel_pass(stage_events, append_events):
        # the first layer's launches with per-stage events (stages back to
        # back). A device spin first (torch's, about half a millisecond) lets
        # the host enqueue the whole pass before the GPU reaches it, so each
        # event pair brackets its kernel's execution, not the host's launch
        # work.
        plan = B.Plan(w.requests, w.block_table, cfg, device=dev, workspace=ws, opts=opts)
        torch.cuda._sleep(SPIN_CYCLES)
        append_events[0].record(stream)
        append(caches[0])
        append_events[1].record(stream)
        forward(plan, caches[0], q, stage_events)
        plan.close()

    for _ in range(args.warmup):
        flush()
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
        flush()
        step()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    host_s = 0.0
    plan_s = []
    for i in range(K):
        flush()
        ev[i][0].record(stream)
        h0 = time.perf_counter()
        t_plan = step()
        host_s += time.perf_counter() - h0
        plan_s.append(t_plan)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    t_end = time.perf_counter() + (0.0 if args.no_clocks else 0.3)
    while time.perf_counter() < t_end:
        flush()
        step()
        torch.cuda.synchronize()
    clk = clocks.stop()
    # per-kernel durations for the roofline: the same launches again, each
    # stage bracketed by its own events (L2 flushed before every pass)
    for i in range(K):
        flush()
        kernel_pass(sev[i], aev[i])
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    stage_ms = {}
    for sname in STAGES:
        si = STAGE_INDEX[sname]
        if info[{"decode": "n_decode_items", "prefill": "n_prefill_items"}[sname]] > 0:
            stage_ms[sname] = statistics.mean(
                sev[i][2 * si].elapsed_time(sev[i][2 * si + 1]) for i in range(K))
    stage_ms["append"] = statistics.mean(a.elapsed_time(b) for a, b in aev)
    ms_step = statistics.mean(step_ms)
    value, total_ms = job_throughput(sum(step_ms), w.total_q, K, world)
    dev_status = int(ws[:4].view(torch.int32).item()) | int(status.item())

    peaks = load_peaks()
    work = stage_work(w, fp8=fp8, prefill_mask=prefill_request_mask(w, cfg, opts))
    if rope:
        work["append_bytes"] = C.rope_append_bytes(w.total_q, s.n_q_heads, s.n_kv_heads,
                                                   s.head_dim)
    names = {"prefill": ("dequant_pages_kernel + prefill_kernel (tcgen05)" if fp8 else
                         "prefill_kernel (tcgen05)"),
             "decode": (("splitkv_fp8t_kernel (few-row form)"
                         if s.head_dim == 128 and 0 < info.get("splitkv_max_rows", 0) <= 8
                         else "splitkv_fp8_kernel") if fp8 else "splitkv_kernel"),
             "append": ("rope_append_kernel" if rope else
                        "kv_append_fp8_kernel" if fp8 else "kv_append_kernel")}
    dominant = max(stage_ms, key=stage_ms.get) if stage_ms else None
    roof = roofline(dominant, stage_ms, work, peaks, names, s.name, fp8)

    res = {"w": w, "info": info, "stage_ms": stage_ms, "ms_step": ms_step, "value": value,
           "total_ms": total_ms, "roof": roof, "work": work, "clk": clk,
           "dev_status": dev_status, "wall": wall, "host_s": host_s,
           "plan_us": statistics.median(plan_s) * 1e6,
           "launches": launches_per_step * K, "layers": L, "peaks": peaks,
           "combined": combined_bound(work, ms_step, peaks, L)}

    # ---- end to end through host buffers
    if main and not args.no_e2e:
        res["e2e"] = measure_e2e(args, w, cfg, opts, dev, ws, info, world, caches, slots,
                                 append_rows, forward, flush, out, lse, stream)
    return res


def measure_e2e(args, w, cfg, opts, dev, ws, info, world, caches, slots, append_rows, forward,
                flush, out, lse, stream):
    """The same step through the public calls with host buffers: each step
    uploads its Q/K/V from pinned memory and downloads O and LSE."""
    import torch

    from continuous_batching_paged_varlen_gb300 import binding as B

    K = args.steps
    q, k_new, v_new = w.q, w.k_new, w.v_new
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
        plan = B.Plan(w.requests, w.block_table, cfg, device=dev, workspace=ws, opts=opts)
        for c in caches:
            append_rows(c, dk, dv, slots)
            forward(plan, c, dq)
        plan.close()
        hout.copy_(out, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    for _ in range(max(3, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e_ms = []
    for i in range(K):
        flush()
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
    # compute stream behind the next step's bulk upload.
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
        for c in caches:
            append_rows(c, b["k"], b["v"], slots)
            forward(plan, c, b["q"], o=b["o"], l=b["l"])
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
    return {"value": world * w.total_q / (piped_ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": piped_ms,
            "timing": "K steps through the public calls, pipelined (each step's Q/K/V "
                      "upload from pinned host memory and its plan on an upload stream, "
                      "append + forward on the compute stream, O/LSE download on a third "
                      "stream; inputs, outputs and workspaces rotate over 3 buffer sets); "
                      "host wall clock over the K steps, synchronised at both ends",
            "serial": {"value": world * w.total_q / (statistics.mean(e_ms) / 1e3),
                       "ms_per_step": statistics.mean(e_ms),
                       "timing": "one step at a time: host wall clock around each step, "
                                 "synchronised, L2 flushed before it"}}


def workload_summary(r):
    """One entry of the line's ``workloads`` object."""
    w = r["w"]
    s = w.spec
    d = {"description": s.description, "q_rows": w.total_q, "requests": w.n_requests,
         "ms_per_step": r["ms_step"], "value": r["value"], "unit": UNIT,
         "stages_ms": r["stage_ms"], "roofline": r["roof"],
         "combined_bound": r["combined"],
         "algorithmic": {"attention_flops": r["work"]["total_flops"],
                         "attention_bytes": r["work"]["total_bytes"],
                         "append_bytes": r["work"]["append_bytes"],
                         "decode_bytes": r["work"]["decode_bytes"],
                         "prefill_flops": r["work"]["prefill_flops"]},
         "plan": {k: r["info"][k] for k in ("n_decode_items", "n_prefill_items", "n_combine",
                                            "n_cascade_groups", "cascade_keys", "kv_chunk")},
         "clocks": r["clk"], "device_status": r["dev_status"], "gpu_launches": r["launches"],
         "plan_host_us": r["plan_us"]}
    if s.shared_prefix:
        stored = C.distinct_kv_positions(w.requests, w.block_table, s.page_size)
        naive = C.naive_kv_positions(w.requests)
        per_pos = C.bytes_per_position(1, s.n_kv_heads, s.head_dim)
        d["prefix"] = {"stored_kv_bytes": stored * per_pos, "naive_kv_bytes": naive * per_pos,
                       "ncu_dram_bytes_per_launch": recorded_traffic("decode", s.name)}
    return d


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

    r = measure(args, args.workload, dev, local, world, main=True)
    w = r["w"]
    work, info, stage_ms, ms_step = r["work"], r["info"], r["stage_ms"], r["ms_step"]
    line = {
        "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 KV + bf16" if args.fp8 else "bf16", "data": "synthetic",
        "config": workload_config_args(w, args, world),
        "roofline": r["roof"], "cpu_baseline": None, "e2e": r.get("e2e"),
        "gpu_launches": r["launches"],
        "clocks": r["clk"],
        "stages_ms": stage_ms,
        "achieved": {"attention_tflops": r["layers"] * work["total_flops"] / (ms_step / 1e3) / 1e12,
                     "attention_hbm_gbs": r["layers"] * work["total_bytes"] / (ms_step / 1e3) / 1e9,
                     "algorithmic_flops_per_step": r["layers"] * work["total_flops"],
                     "algorithmic_bytes_per_step": r["layers"] * (work["total_bytes"]
                                                                  + work["append_bytes"]),
                     "append_hbm_gbs": work["append_bytes"] / (stage_ms["append"] / 1e3) / 1e9},
        "combined_bound": r["combined"],
        "plan": info, "device_status": r["dev_status"], "wall_s_timed_region": r["wall"],
        # host time to enqueue one step (append, plan + upload, forward, through
        # the Python binding); a step shorter than this on the device is
        # host-bound, the GPU waiting for its launches
        "host_enqueue_us_per_step": r["host_s"] / args.steps * 1e6,
        "plan_host_us": r["plan_us"],
    }
    dev_status = r["dev_status"]
    cpu_w = w
    del r
    torch.cuda.empty_cache()

    plain = not (args.fp8 or args.rope or args.max_requests or args.disable_cascade
                 or args.layers > 1 or args.prefill_ctas or args.kv_chunk)
    if args.workload == DEFAULT_WORKLOAD and plain and not args.no_workloads:
        extra = {}
        for name in LINE_WORKLOADS:
            x = measure(args, name, dev, local, world, main=False)
            extra[name] = workload_summary(x)
            dev_status |= x["dev_status"]
            line["gpu_launches"] += x["launches"]
            del x
            torch.cuda.empty_cache()
        line["workloads"] = extra

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(cpu_w, args.cpu_seconds, fp8=args.fp8)
        if args.layers > 1:  # the oracle ran one layer; the line's step runs every layer
            cb["value"] /= args.layers
            cb["one_thread"]["value"] /= args.layers
            cb["sample"] += f"; rate divided by {args.layers} layers"
        line["cpu_baseline"] = cb
    line["device_status"] = dev_status
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
