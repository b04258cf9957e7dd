"""Thin ctypes binding of ``libmb.so`` (the C ABI in ``include/mb.h``).

Only argument marshalling happens here: every step of the attention path
runs in the library's CUDA kernels. The library is loaded lazily by
``lib()``, which raises when it has not been built -- there is no fallback.
PyTorch supplies device memory and streams; tensors are passed by pointer.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmb.so")
ABI_VERSION = 3  # MB_ABI_VERSION of include/mb.h the structures below mirror

MB_OK = 0
STATUS_NAMES = {0: "MB_OK", 1: "MB_ERR_INVALID_ARG", 2: "MB_ERR_SHAPE",
                3: "MB_ERR_UNSUPPORTED", 4: "MB_ERR_WORKSPACE", 5: "MB_ERR_CUDA",
                6: "MB_ERR_TIMEOUT", 7: "MB_ERR_DEVICE_INDEX", 8: "MB_ERR_SHARED_PAGE"}
MB_ERR_WORKSPACE = 4
MB_ERR_TIMEOUT = 6
MB_ERR_DEVICE_INDEX = 7
MB_ERR_SHARED_PAGE = 8
STAGE_DECODE, STAGE_COMBINE, STAGE_PREFILL, NUM_STAGES = 0, 1, 2, 3


class MBError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


class Request(ctypes.Structure):
    _fields_ = [("q_start", ctypes.c_int32), ("q_end", ctypes.c_int32),
                ("kv_length", ctypes.c_int32)]


class Config(ctypes.Structure):
    _fields_ = [("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("max_blocks_per_req", ctypes.c_int32),
                ("scale", ctypes.c_float)]


class PlanOptions(ctypes.Structure):
    _fields_ = [("prefill_min_rows", ctypes.c_int32), ("kv_chunk", ctypes.c_int32),
                ("disable_cascade", ctypes.c_int32), ("target_ctas", ctypes.c_int32),
                ("prefill_ctas", ctypes.c_int32), ("fp8_cache", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("n_decode_items", ctypes.c_int32), ("n_decode_rows", ctypes.c_int32),
                ("n_prefill_items", ctypes.c_int32), ("n_combine", ctypes.c_int32),
                ("n_partials", ctypes.c_int32), ("n_cascade_groups", ctypes.c_int32),
                ("cascade_keys", ctypes.c_int32), ("kv_chunk", ctypes.c_int32),
                ("total_q", ctypes.c_int32), ("n_launches", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_size_t), ("metadata_bytes", ctypes.c_size_t),
                ("prefill_ctas", ctypes.c_int32), ("staged_pages", ctypes.c_int32),
                ("splitkv_copies", ctypes.c_int32), ("splitkv_max_rows", ctypes.c_int32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class SchedConfig(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_blocks_per_req", ctypes.c_int32), ("token_budget", ctypes.c_int32),
                ("max_running", ctypes.c_int32), ("decode_rows", ctypes.c_int32)]


class SchedStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("n_reqs", "total_q", "n_prefill", "n_decode", "n_preempted", "n_prefix_hits",
                 "n_waiting", "n_running", "n_finished", "free_pages")]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


SCHED_STATES = {0: "waiting", 1: "prefill", 2: "decode", 3: "finished"}

_lib = None
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_pi32 = ctypes.POINTER(ctypes.c_int32)


def lib():
    """The loaded library; raises if ``libmb.so`` is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (there is no fallback path)")
    L = ctypes.CDLL(LIB_PATH)
    L.mb_abi_version.restype = _i32
    if L.mb_abi_version() != ABI_VERSION:
        raise RuntimeError(f"{LIB_PATH} has ABI version {L.mb_abi_version()}, the binding "
                           f"expects {ABI_VERSION}: rebuild it")
    L.mb_status_string.restype = ctypes.c_char_p
    L.mb_status_string.argtypes = [ctypes.c_int]
    L.mb_slot_mapping.restype = ctypes.c_int
    L.mb_slot_mapping.argtypes = [_vp, _i32, _vp, ctypes.POINTER(Config), _vp, _i32]
    L.mb_kv_append.restype = ctypes.c_int
    L.mb_kv_append.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, ctypes.POINTER(Config), _vp, _vp]
    L.mb_kv_append_fp8.restype = ctypes.c_int
    L.mb_kv_append_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                   ctypes.POINTER(Config), _vp, _vp]
    L.mb_attn_forward_fp8.restype = ctypes.c_int
    L.mb_attn_forward_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    L.mb_attn_forward_fp8_timed.restype = ctypes.c_int
    L.mb_attn_forward_fp8_timed.argtypes = [_vp] * 11
    L.mb_positions.restype = ctypes.c_int
    L.mb_positions.argtypes = [_vp, _i32, _vp, _i32]
    L.mb_rope_table.restype = ctypes.c_int
    L.mb_rope_table.argtypes = [_vp, _i32, _i32, ctypes.c_float]
    L.mb_rope_kv_append.restype = ctypes.c_int
    L.mb_rope_kv_append.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32,
                                    ctypes.POINTER(Config), _vp, _vp]
    L.mb_attn_plan.restype = ctypes.c_int
    L.mb_attn_plan.argtypes = [_vp, _i32, _vp, ctypes.POINTER(Config), _vp,
                               ctypes.POINTER(ctypes.c_size_t), _vp, ctypes.POINTER(_vp)]
    L.mb_attn_plan_ex.restype = ctypes.c_int
    L.mb_attn_plan_ex.argtypes = [_vp, _i32, _vp, ctypes.POINTER(Config),
                                  ctypes.POINTER(PlanOptions), _vp,
                                  ctypes.POINTER(ctypes.c_size_t), _vp, ctypes.POINTER(_vp)]
    L.mb_attn_plan_host.restype = ctypes.c_int
    L.mb_attn_plan_host.argtypes = [_vp, _i32, _vp, ctypes.POINTER(Config),
                                    ctypes.POINTER(PlanOptions), ctypes.POINTER(_vp)]
    L.mb_attn_forward.restype = ctypes.c_int
    L.mb_attn_forward.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    L.mb_attn_forward_timed.restype = ctypes.c_int
    L.mb_attn_forward_timed.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    L.mb_plan_info.restype = ctypes.c_int
    L.mb_plan_info.argtypes = [_vp, ctypes.POINTER(PlanInfo)]
    L.mb_plan_export_metadata.restype = ctypes.c_int
    L.mb_plan_export_metadata.argtypes = [_vp, _vp, ctypes.c_size_t]
    L.mb_plan_layout.restype = ctypes.c_int
    L.mb_plan_layout.argtypes = [_vp, ctypes.POINTER(ctypes.c_size_t)]
    L.mb_attn_destroy.restype = ctypes.c_int
    L.mb_attn_destroy.argtypes = [_vp]
    L.mb_check_append_targets.restype = ctypes.c_int
    L.mb_check_append_targets.argtypes = [_vp, _i32, _vp, ctypes.POINTER(Config),
                                          ctypes.POINTER(_i32)]
    L.mb_selftest_wait_timeout.restype = ctypes.c_int
    L.mb_selftest_wait_timeout.argtypes = [_vp, _vp]
    L.mb_attn_forward_noalloc.restype = ctypes.c_int
    L.mb_attn_forward_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    L.mb_sched_create.restype = ctypes.c_int
    L.mb_sched_create.argtypes = [ctypes.POINTER(SchedConfig), ctypes.POINTER(_vp)]
    L.mb_sched_destroy.restype = ctypes.c_int
    L.mb_sched_destroy.argtypes = [_vp]
    L.mb_sched_add.restype = ctypes.c_int
    L.mb_sched_add.argtypes = [_vp, _i32, _i32, _i32, _i32, _pi32]
    L.mb_sched_step.restype = ctypes.c_int
    L.mb_sched_step.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32,
                                ctypes.POINTER(SchedStats)]
    L.mb_sched_commit.restype = ctypes.c_int
    L.mb_sched_commit.argtypes = [_vp, _vp, _i32, _pi32]
    L.mb_sched_page_refs.restype = ctypes.c_int
    L.mb_sched_page_refs.argtypes = [_vp, _vp, _i32]
    L.mb_sched_request_info.restype = ctypes.c_int
    L.mb_sched_request_info.argtypes = [_vp, _i32, _vp]
    _lib = L
    return L


def check(status: int, what: str):
    if status != MB_OK:
        raise MBError(status, what)


def config(n_q_heads, n_kv_heads, head_dim, page_size, num_pages, max_blocks_per_req,
           scale=0.0) -> Config:
    return Config(n_q_heads, n_kv_heads, head_dim, page_size, num_pages,
                  max_blocks_per_req, float(scale or 0.0))


def options(prefill_min_rows=0, kv_chunk=0, disable_cascade=0, target_ctas=0,
            prefill_ctas=0, fp8_cache=0) -> PlanOptions:
    return PlanOptions(prefill_min_rows, kv_chunk, disable_cascade, target_ctas, prefill_ctas,
                       fp8_cache)


def _host_i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def slot_mapping(requests, block_table, cfg: Config, total_q: int) -> np.ndarray:
    """``mb_slot_mapping``: int32 slot of every flat new row (-1 if uncovered)."""
    reqs = _host_i32(requests).reshape(-1, 3)
    bt = _host_i32(block_table)
    out = np.empty(max(total_q, 1), dtype=np.int32)
    check(lib().mb_slot_mapping(reqs.ctypes.data, reqs.shape[0], bt.ctypes.data,
                                ctypes.byref(cfg), out.ctypes.data, total_q),
          "mb_slot_mapping")
    return out[:total_q]


def check_append_targets(requests, block_table, cfg: Config):
    """``mb_check_append_targets``: (status, first offending request or -1);
    MB_ERR_SHARED_PAGE when a new row would land in a page another request
    also maps."""
    reqs = _host_i32(requests).reshape(-1, 3)
    bt = _host_i32(block_table)
    bad = _i32(-1)
    st = lib().mb_check_append_targets(reqs.ctypes.data, reqs.shape[0], bt.ctypes.data,
                                       ctypes.byref(cfg), ctypes.byref(bad))
    return int(st), int(bad.value)


def selftest_wait_timeout(status, stream=None):
    """``mb_selftest_wait_timeout``: one CTA's bounded wait on an mbarrier
    nothing completes runs out; it sets bit ``1 << MB_ERR_TIMEOUT`` in
    ``status`` (device int32) and returns. Read the status after a sync."""
    check(lib().mb_selftest_wait_timeout(_ptr(status), _stream_ptr(stream)),
          "mb_selftest_wait_timeout")


def kv_append(k_cache, v_cache, k_new, v_new, slots, cfg: Config, status=None, stream=None):
    """``mb_kv_append`` on torch tensors (``slots``: int32 device tensor)."""
    T = int(slots.numel())
    check(lib().mb_kv_append(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
                             _ptr(slots), T, ctypes.byref(cfg), _ptr(status),
                             _stream_ptr(stream) if T else None),
          "mb_kv_append")


def positions(requests, total_q: int) -> np.ndarray:
    """``mb_positions``: logical position of every new row (host int32)."""
    reqs = _host_i32(requests).reshape(-1, 3)
    out = np.empty(max(total_q, 1), dtype=np.int32)
    check(lib().mb_positions(reqs.ctypes.data, reqs.shape[0], out.ctypes.data, total_q),
          "mb_positions")
    return out[:total_q]


def rope_table(max_position: int, head_dim: int, base: float = 10000.0) -> np.ndarray:
    """``mb_rope_table``: host fp32 [max_position, head_dim] angle table."""
    out = np.empty((max_position, head_dim), dtype=np.float32)
    check(lib().mb_rope_table(out.ctypes.data, max_position, head_dim, float(base)),
          "mb_rope_table")
    return out


def kv_append_fp8(k_codes, v_codes, k_scale, v_scale, k_new, v_new, slots, cfg: Config,
                  status=None, stream=None):
    """``mb_kv_append_fp8`` on torch tensors: quantizes each (token, KV head)
    row of ``k_new`` / ``v_new`` (bf16) into the e4m3 code caches (uint8) and
    their fp32 per-row scales."""
    T = int(slots.numel())
    check(lib().mb_kv_append_fp8(_ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(v_scale),
                                 _ptr(k_new), _ptr(v_new), _ptr(slots), T, ctypes.byref(cfg),
                                 _ptr(status), _stream_ptr(stream) if T else None),
          "mb_kv_append_fp8")


def rope_kv_append(q, k_cache, v_cache, k_new, v_new, positions_dev, slots, cos_sin,
                   cfg: Config, status=None, stream=None):
    """``mb_rope_kv_append`` on torch tensors: rotates ``q`` in place, writes the
    rotated ``k_new`` and ``v_new`` into the caches (``positions_dev``,
    ``slots``: int32 device tensors; ``cos_sin``: fp32 device table)."""
    T = int(slots.numel())
    check(lib().mb_rope_kv_append(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_new),
                                  _ptr(v_new), _ptr(positions_dev), _ptr(slots), T,
                                  _ptr(cos_sin), int(cos_sin.shape[0]) if cos_sin is not None else 0,
                                  ctypes.byref(cfg), _ptr(status),
                                  _stream_ptr(stream) if T else None),
          "mb_rope_kv_append")


class HostPlan:
    """A plan built on the host only (``mb_attn_plan_host``), for inspection."""

    def __init__(self, requests, block_table, cfg: Config, opts: Optional[PlanOptions] = None):
        self.reqs = _host_i32(requests).reshape(-1, 3)
        self.bt = _host_i32(block_table)
        self.cfg = cfg
        h = ctypes.c_void_p()
        check(lib().mb_attn_plan_host(self.reqs.ctypes.data, self.reqs.shape[0],
                                      self.bt.ctypes.data, ctypes.byref(cfg),
                                      ctypes.byref(opts) if opts else None, ctypes.byref(h)),
              "mb_attn_plan_host")
        self._h = h

    @property
    def info(self) -> PlanInfo:
        inf = PlanInfo()
        check(lib().mb_plan_info(self._h, ctypes.byref(inf)), "mb_plan_info")
        return inf

    def layout(self):
        arr = (ctypes.c_size_t * 6)()
        check(lib().mb_plan_layout(self._h, arr), "mb_plan_layout")
        return list(arr)

    def metadata(self) -> bytes:
        n = self.info.metadata_bytes
        buf = (ctypes.c_uint8 * n)()
        check(lib().mb_plan_export_metadata(self._h, buf, n), "mb_plan_export_metadata")
        return bytes(buf)

    def close(self):
        if self._h:
            lib().mb_attn_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def forward_noalloc(host_plan: "HostPlan", q, k_cache, v_cache, block_table_dev, out, lse=None,
                    status=None, stream=None):
    """``mb_attn_forward_noalloc``: run a host-only plan with the library's
    static scratch array instead of a workspace (for callers that must not
    allocate device memory; see include/mb.h)."""
    check(lib().mb_attn_forward_noalloc(host_plan._h, _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(block_table_dev), _ptr(out), _ptr(lse),
                                        _ptr(status), _stream_ptr(stream)),
          "mb_attn_forward_noalloc")


class Plan:
    """``mb_attn_plan`` + a caller-owned (torch) workspace; ``forward`` runs
    ``mb_attn_forward`` on the given stream."""

    def __init__(self, requests, block_table, cfg: Config, device="cuda",
                 opts: Optional[PlanOptions] = None, stream=None, workspace=None):
        import torch
        self.reqs = _host_i32(requests).reshape(-1, 3)
        self.bt = _host_i32(block_table)
        self.cfg = cfg
        L = lib()
        o = ctypes.byref(opts) if opts else None
        h = ctypes.c_void_p()
        st = MB_ERR_WORKSPACE
        if workspace is not None:
            # a caller's workspace is tried first: a plan that fits needs no
            # size query (the planner runs once)
            nb = ctypes.c_size_t(workspace.numel())
            st = L.mb_attn_plan_ex(self.reqs.ctypes.data, self.reqs.shape[0],
                                   self.bt.ctypes.data, ctypes.byref(cfg), o, _ptr(workspace),
                                   ctypes.byref(nb), _stream_ptr(stream), ctypes.byref(h))
        if st == MB_ERR_WORKSPACE:
            nbytes = ctypes.c_size_t(0)
            check(L.mb_attn_plan_ex(self.reqs.ctypes.data, self.reqs.shape[0],
                                    self.bt.ctypes.data, ctypes.byref(cfg), o, None,
                                    ctypes.byref(nbytes), None, None),
                  "mb_attn_plan (size query)")
            workspace = torch.empty(max(int(nbytes.value), 256), dtype=torch.uint8,
                                    device=device)
            nb = ctypes.c_size_t(workspace.numel())
            st = L.mb_attn_plan_ex(self.reqs.ctypes.data, self.reqs.shape[0],
                                   self.bt.ctypes.data, ctypes.byref(cfg), o, _ptr(workspace),
                                   ctypes.byref(nb), _stream_ptr(stream), ctypes.byref(h))
        check(st, "mb_attn_plan")
        self.workspace = workspace
        self._h = h
        self.workspace_bytes = int(self.info.workspace_bytes)

    @property
    def info(self) -> PlanInfo:
        inf = PlanInfo()
        check(lib().mb_plan_info(self._h, ctypes.byref(inf)), "mb_plan_info")
        return inf

    def forward(self, q, k_cache, v_cache, block_table_dev, out, lse=None, stream=None,
                events=None):
        L = lib()
        if events is None:
            st = L.mb_attn_forward(self._h, _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(block_table_dev), _ptr(out), _ptr(lse),
                                   _stream_ptr(stream))
        else:
            arr = (ctypes.c_void_p * (2 * NUM_STAGES))(
                *[None if e is None else ctypes.c_void_p(e.cuda_event) for e in events])
            st = L.mb_attn_forward_timed(self._h, _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                         _ptr(block_table_dev), _ptr(out), _ptr(lse),
                                         _stream_ptr(stream), arr)
        check(st, "mb_attn_forward")

    def forward_fp8(self, q, k_codes, v_codes, k_scale, v_scale, block_table_dev, out,
                    lse=None, stream=None, events=None):
        """``mb_attn_forward_fp8``: attention over an fp8 (e4m3) cache; the plan
        must hold no prefill items (plan with ``prefill_min_rows=-1``)."""
        L = lib()
        args = (self._h, _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(v_scale),
                _ptr(block_table_dev), _ptr(out), _ptr(lse), _stream_ptr(stream))
        if events is None:
            st = L.mb_attn_forward_fp8(*args)
        else:
            arr = (ctypes.c_void_p * (2 * NUM_STAGES))(
                *[None if e is None else ctypes.c_void_p(e.cuda_event) for e in events])
            st = L.mb_attn_forward_fp8_timed(*args, arr)
        check(st, "mb_attn_forward_fp8")

    def device_status(self) -> int:
        """Device error flags of this plan's workspace (synchronises)."""
        return int(self.workspace[:4].view(dtype=__import__("torch").int32).item())

    def close(self):
        if getattr(self, "_h", None):
            lib().mb_attn_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Iteration:
    """One built iteration of ``Scheduler.step``: host arrays shaped for the
    library's calls (``requests`` [n, 3] triples, ``ids`` [n], ``block_table``
    [n, max_blocks], ``slots`` and ``positions`` [total_q]) and the counters."""

    def __init__(self, requests, ids, block_table, slots, positions, stats):
        self.requests, self.ids, self.block_table = requests, ids, block_table
        self.slots, self.positions, self.stats = slots, positions, stats

    @property
    def total_q(self) -> int:
        return int(self.stats["total_q"])


class Scheduler:
    """The host iteration builder of ``include/mb_sched.h`` (``mb_sched_*``)."""

    def __init__(self, num_pages, page_size, max_blocks_per_req, token_budget, max_running=0,
                 decode_rows=1):
        self.cfg = SchedConfig(num_pages, page_size, max_blocks_per_req, token_budget,
                               max_running, decode_rows)
        h = _vp()
        check(lib().mb_sched_create(ctypes.byref(self.cfg), ctypes.byref(h)), "mb_sched_create")
        self._h = h
        self.n_added = 0

    def add(self, prompt_len, max_new_tokens, prefix_id=-1, prefix_len=0) -> int:
        rid = ctypes.c_int32()
        check(lib().mb_sched_add(self._h, prompt_len, max_new_tokens, prefix_id, prefix_len,
                                 ctypes.byref(rid)), "mb_sched_add")
        self.n_added += 1
        return int(rid.value)

    def step(self) -> Iteration:
        cap_r = max(1, self.n_added)
        cap_q = max(1, self.cfg.token_budget)
        mb = self.cfg.max_blocks_per_req
        reqs = np.zeros((cap_r, 3), np.int32)
        ids = np.zeros(cap_r, np.int32)
        bt = np.zeros((cap_r, mb), np.int32)
        slots = np.zeros(cap_q, np.int32)
        pos = np.zeros(cap_q, np.int32)
        st = SchedStats()
        check(lib().mb_sched_step(self._h, reqs.ctypes.data, ids.ctypes.data, bt.ctypes.data,
                                  slots.ctypes.data, pos.ctypes.data, cap_r, cap_q,
                                  ctypes.byref(st)), "mb_sched_step")
        n, q = st.n_reqs, st.total_q
        return Iteration(reqs[:n].copy(), ids[:n].copy(), bt[:n].copy(), slots[:q].copy(),
                         pos[:q].copy(), st.as_dict())

    def commit(self) -> list:
        out = np.zeros(max(1, self.n_added), np.int32)
        n = ctypes.c_int32()
        check(lib().mb_sched_commit(self._h, out.ctypes.data, out.size, ctypes.byref(n)),
              "mb_sched_commit")
        return out[:n.value].tolist()

    def page_refs(self) -> np.ndarray:
        out = np.zeros(self.cfg.num_pages, np.int32)
        check(lib().mb_sched_page_refs(self._h, out.ctypes.data, out.size), "mb_sched_page_refs")
        return out

    def request_info(self, rid) -> dict:
        out = np.zeros(8, np.int32)
        check(lib().mb_sched_request_info(self._h, rid, out.ctypes.data), "mb_sched_request_info")
        keys = ("state", "computed", "generated", "pages", "preemptions", "prompt_len",
                "max_new_tokens", "prefix_id")
        d = dict(zip(keys, out.tolist()))
        d["state"] = SCHED_STATES[d["state"]]
        return d

    def close(self):
        if self._h:
            lib().mb_sched_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
