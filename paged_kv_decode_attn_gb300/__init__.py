"""Python binding of the oxd C ABI (``include/oxd.h``) -- argument marshalling only.

Every step of the decode path runs in ``lib/liboxd.so`` (built from ``csrc/``
by :func:`build`). This module loads that library with ctypes, turns tensors
into device pointers and statuses into exceptions, and nothing else; there is
no Python or CPU fallback. If the library is missing, importing works but
every call raises :class:`LibraryNotBuilt`.

The functions keep the C names:

* :func:`oxd_paged_decode_plan` -> :class:`Plan` (owns the opaque handle)
* :func:`oxd_paged_decode_run`, :func:`oxd_plan_bind_workspace`
* :func:`oxd_merge_states`
* :func:`oxd_rope_append` (fused rotary embedding + paged KV append)
* :func:`oxd_plan_get_info`, :func:`oxd_plan_set_timing_events`,
  :func:`oxd_plan_destroy`, :func:`oxd_read_device_status`,
  :func:`oxd_status_string`, :func:`oxd_device_status_string`, :func:`oxd_version`

Tensor arguments may be torch tensors (their ``data_ptr()`` is passed) or
plain integers (raw addresses). Streams may be a ``torch.cuda.Stream``, a raw
``cudaStream_t`` integer, or ``None`` (torch's current stream on the tensors'
device when torch is importable, else the legacy default stream).
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from .build import LIB as LIB_PATH
from .build import build

__all__ = [
    "OXD_OK", "OXD_LAYOUT_NHD", "OXD_LAYOUT_HND", "OxdError", "LibraryNotBuilt", "Desc",
    "PlanInfo", "Plan", "build", "lib", "oxd_paged_decode_plan", "oxd_paged_decode_run",
    "oxd_paged_decode_run_static_workspace", "oxd_read_static_workspace_status",
    "oxd_plan_bind_workspace", "oxd_merge_states", "oxd_plan_get_info", "oxd_plan_set_timing_events", "oxd_plan_destroy",
    "oxd_read_device_status", "oxd_status_string", "oxd_device_status_string", "oxd_version",
    "oxd_rope_append", "RopeAppendDesc", "make_rope_append_desc", "EXPORTED_SYMBOLS",
    "PrefillDesc", "PrefillPlanInfo", "PrefillPlan", "make_prefill_desc",
    "oxd_paged_prefill_plan", "oxd_paged_prefill_run", "oxd_prefill_plan_bind_workspace",
    "oxd_prefill_plan_get_info", "oxd_prefill_plan_set_timing_events",
    "oxd_prefill_plan_destroy",
]

OXD_OK = 0
OXD_ERR_INVALID_ARGUMENT = 1
OXD_ERR_UNSUPPORTED = 2
OXD_ERR_ALIGNMENT = 3
OXD_ERR_ALIAS = 4
OXD_ERR_WORKSPACE_TOO_SMALL = 5
OXD_ERR_PLAN_MISMATCH = 6
OXD_ERR_CUDA = 7
OXD_ERR_DEVICE_STATUS = 8
OXD_ERR_NO_MEMORY = 9

OXD_LAYOUT_NHD = 0
OXD_LAYOUT_HND = 1

OXD_DEVICE_OK = 0
OXD_DEVICE_BAD_PAGE = 1
OXD_DEVICE_PLAN_MISMATCH = 2
OXD_DEVICE_WAIT_TIMEOUT = 3
OXD_DEVICE_SHARED_PAGE = 4
OXD_DEVICE_BAD_POSITION = 5

EXPORTED_SYMBOLS = (
    "oxd_paged_decode_plan", "oxd_paged_decode_run", "oxd_merge_states", "oxd_plan_get_info",
    "oxd_plan_set_timing_events", "oxd_plan_destroy", "oxd_read_device_status",
    "oxd_status_string", "oxd_device_status_string", "oxd_version",
    "oxd_paged_decode_run_static_workspace", "oxd_read_static_workspace_status",
    "oxd_plan_bind_workspace", "oxd_rope_append",
    "oxd_paged_prefill_plan", "oxd_paged_prefill_run", "oxd_prefill_plan_bind_workspace",
    "oxd_prefill_plan_get_info", "oxd_prefill_plan_set_timing_events",
    "oxd_prefill_plan_destroy",
)


class LibraryNotBuilt(RuntimeError):
    """liboxd.so is not built (call paged_kv_decode_attn_gb300.build())."""


class OxdError(RuntimeError):
    def __init__(self, func: str, status: int, detail: str = ""):
        self.status = status
        self.func = func
        msg = f"{func}: {oxd_status_string(status)} ({status})"
        super().__init__(msg + (f": {detail}" if detail else ""))


class Desc(ctypes.Structure):
    """``oxd_paged_decode_desc``."""

    _fields_ = [
        ("batch", ctypes.c_int32), ("num_qo_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("layout", ctypes.c_int32),
        ("num_pages", ctypes.c_int64), ("max_splits", ctypes.c_int32),
        ("force_splits", ctypes.c_int32), ("num_sms", ctypes.c_int32),
        ("tensor_path", ctypes.c_int32), ("shared_prefix_tokens", ctypes.c_int32),
        ("share_group", ctypes.c_int32), ("pdl", ctypes.c_int32),
        ("wait_timeout_ns", ctypes.c_int64),
    ]


class PlanInfo(ctypes.Structure):
    """``oxd_plan_info``."""

    _fields_ = [
        ("num_work_items", ctypes.c_int32), ("num_split_requests", ctypes.c_int32),
        ("max_chunks", ctypes.c_int32), ("chunk_pages", ctypes.c_int32),
        ("num_slots", ctypes.c_int32), ("kernel_variant", ctypes.c_int32),
        ("grid_ctas", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32),
        ("num_sms", ctypes.c_int32), ("launches_per_run", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_int64), ("upload_bytes", ctypes.c_int64),
        ("total_kv_tokens", ctypes.c_int64), ("cascade_units", ctypes.c_int32),
        ("cascade_requests", ctypes.c_int32), ("shared_kv_tokens", ctypes.c_int64),
        ("cluster_size", ctypes.c_int32), ("reserved", ctypes.c_int32),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


_lock = threading.Lock()
_lib = None


class RopeAppendDesc(ctypes.Structure):
    """``oxd_rope_append_desc``."""

    _fields_ = [
        ("num_tokens", ctypes.c_int32), ("batch", ctypes.c_int32),
        ("num_qo_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("layout", ctypes.c_int32), ("num_indices", ctypes.c_int32),
        ("num_pages", ctypes.c_int64), ("rope_theta", ctypes.c_double),
        ("reserved", ctypes.c_int32 * 2),
    ]


class PrefillDesc(ctypes.Structure):
    """``oxd_paged_prefill_desc``."""

    _fields_ = [
        ("batch", ctypes.c_int32), ("num_qo_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("layout", ctypes.c_int32),
        ("num_pages", ctypes.c_int64), ("max_splits", ctypes.c_int32),
        ("num_sms", ctypes.c_int32), ("wait_timeout_ns", ctypes.c_int64),
        ("tile_rows", ctypes.c_int32), ("reserved", ctypes.c_int32),
    ]


class PrefillPlanInfo(ctypes.Structure):
    """``oxd_prefill_plan_info``."""

    _fields_ = [
        ("tile_tokens", ctypes.c_int32), ("num_tiles", ctypes.c_int32),
        ("num_units", ctypes.c_int32), ("num_split_tiles", ctypes.c_int32),
        ("max_pieces", ctypes.c_int32), ("num_merge_rows", ctypes.c_int32),
        ("launches_per_run", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32),
        ("num_sms", ctypes.c_int32), ("tile_rows", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_int64), ("total_q_tokens", ctypes.c_int64),
        ("total_kv_tokens", ctypes.c_int64), ("causal_pairs", ctypes.c_int64),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


def make_prefill_desc(batch, num_qo_heads, num_kv_heads, page_size, layout, num_pages,
                      head_dim=128, max_splits=0, num_sms=0, wait_timeout_ns=0,
                      tile_rows=0) -> PrefillDesc:
    """Convenience constructor; ``layout`` may be "NHD"/"HND" or 0/1; ``tile_rows``
    0 lets the planner pick 128- or 256-row tiles."""
    if isinstance(layout, str):
        layout = {"NHD": OXD_LAYOUT_NHD, "HND": OXD_LAYOUT_HND}[layout]
    return PrefillDesc(batch, num_qo_heads, num_kv_heads, head_dim, page_size, layout, num_pages,
                       max_splits, num_sms, wait_timeout_ns, tile_rows, 0)


def make_rope_append_desc(num_tokens, batch, num_qo_heads, num_kv_heads, page_size, layout,
                          num_pages, num_indices, rope_theta=10000.0,
                          head_dim=128) -> RopeAppendDesc:
    if isinstance(layout, str):
        layout = {"NHD": OXD_LAYOUT_NHD, "HND": OXD_LAYOUT_HND}[layout]
    return RopeAppendDesc(num_tokens, batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                          layout, num_indices, num_pages, rope_theta,
                          (ctypes.c_int32 * 2)(0, 0))


def lib():
    """The loaded liboxd.so with its signatures declared."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise LibraryNotBuilt(f"{LIB_PATH} is missing; run "
                                      "paged_kv_decode_attn_gb300.build()")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
            L.oxd_paged_decode_plan.argtypes = [ctypes.POINTER(Desc), vp, vp, ctypes.c_int,
                                                ctypes.POINTER(vp), ctypes.POINTER(sz)]
            L.oxd_paged_decode_run.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp,
                                               vp, vp, sz, vp]
            L.oxd_paged_decode_run_static_workspace.argtypes = [
                vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp]
            L.oxd_merge_states.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp]
            L.oxd_plan_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
            L.oxd_plan_set_timing_events.argtypes = [vp, vp, vp]
            L.oxd_plan_bind_workspace.argtypes = [vp, vp, sz, vp]
            L.oxd_rope_append.argtypes = [ctypes.POINTER(RopeAppendDesc)] + [vp] * 12 + [sz, vp]
            L.oxd_plan_destroy.argtypes = [vp]
            L.oxd_paged_prefill_plan.argtypes = [ctypes.POINTER(PrefillDesc), vp, vp, vp,
                                                 ctypes.c_int, vp, vp]
            L.oxd_paged_prefill_run.argtypes = [vp] * 8 + [ctypes.c_float, vp, vp, vp, sz, vp]
            L.oxd_prefill_plan_bind_workspace.argtypes = [vp, vp, sz, vp]
            L.oxd_prefill_plan_get_info.argtypes = [vp, ctypes.POINTER(PrefillPlanInfo)]
            L.oxd_prefill_plan_set_timing_events.argtypes = [vp, vp, vp]
            L.oxd_prefill_plan_destroy.argtypes = [vp]
            L.oxd_read_device_status.argtypes = [vp, vp, ctypes.POINTER(i32)]
            L.oxd_read_static_workspace_status.argtypes = [vp, ctypes.POINTER(i32)]
            for f in ("oxd_paged_decode_plan", "oxd_paged_decode_run",
                      "oxd_paged_decode_run_static_workspace",
                      "oxd_read_static_workspace_status", "oxd_merge_states",
                      "oxd_plan_get_info", "oxd_plan_set_timing_events", "oxd_plan_destroy",
                      "oxd_read_device_status", "oxd_plan_bind_workspace", "oxd_rope_append",
                      "oxd_paged_prefill_plan", "oxd_paged_prefill_run",
                      "oxd_prefill_plan_bind_workspace", "oxd_prefill_plan_get_info",
                      "oxd_prefill_plan_set_timing_events", "oxd_prefill_plan_destroy"):
                getattr(L, f).restype = ctypes.c_int
            L.oxd_status_string.argtypes = [ctypes.c_int]
            L.oxd_status_string.restype = ctypes.c_char_p
            L.oxd_device_status_string.argtypes = [i32]
            L.oxd_device_status_string.restype = ctypes.c_char_p
            L.oxd_version.argtypes = []
            L.oxd_version.restype = ctypes.c_char_p
            _lib = L
    return _lib


# ------------------------------------------------------------------ marshalling helpers

def _addr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x).__name__}")


def _stream(stream, like=None):
    if stream is None:
        try:
            import torch
        except ImportError:
            return None
        if like is not None and hasattr(like, "device") and like.device.type == "cuda":
            return torch.cuda.current_stream(like.device).cuda_stream
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _event(ev):
    if ev is None:
        return None
    if isinstance(ev, int):
        return ev
    return ev.cuda_event


def _check(func, status, detail=""):
    if status != OXD_OK:
        raise OxdError(func, status, detail)


# ------------------------------------------------------------------ ABI functions

def oxd_version() -> str:
    return lib().oxd_version().decode()


def oxd_status_string(status: int) -> str:
    try:
        return lib().oxd_status_string(int(status)).decode()
    except LibraryNotBuilt:
        return f"status {status}"


def oxd_device_status_string(code: int) -> str:
    return lib().oxd_device_status_string(int(code)).decode()


class Plan:
    """Owns an ``oxd_plan`` handle (destroyed on :meth:`destroy` or garbage collection)."""

    def __init__(self, handle: int, workspace_bytes: int, desc: Desc):
        self.handle = handle
        self.workspace_bytes = workspace_bytes
        self.desc = desc

    @property
    def info(self) -> PlanInfo:
        return oxd_plan_get_info(self)

    def destroy(self):
        if self.handle:
            _check("oxd_plan_destroy", lib().oxd_plan_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            if self.handle:
                lib().oxd_plan_destroy(self.handle)
                self.handle = None
        except Exception:
            pass


def _handle(plan):
    return plan.handle if isinstance(plan, (Plan, PrefillPlan)) else plan


def oxd_paged_decode_plan(desc: Desc, indptr_host, last_page_len_host, device: int = 0) -> Plan:
    """Plan a decode batch from host block tables; returns a :class:`Plan`."""
    indptr = np.ascontiguousarray(np.asarray(indptr_host), dtype=np.int32)
    last = np.ascontiguousarray(np.asarray(last_page_len_host), dtype=np.int32)
    if indptr.shape != (desc.batch + 1,) or last.shape != (desc.batch,):
        raise OxdError("oxd_paged_decode_plan", OXD_ERR_INVALID_ARGUMENT,
                       "indptr must be [batch+1] and last_page_len [batch]")
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    st = lib().oxd_paged_decode_plan(ctypes.byref(desc), indptr.ctypes.data, last.ctypes.data,
                                     int(device), ctypes.byref(h), ctypes.byref(ws))
    _check("oxd_paged_decode_plan", st)
    return Plan(h.value, ws.value, desc)


def oxd_paged_decode_run(plan, q, k_pages, v_pages, indptr, indices, last_page_len, sm_scale,
                         out, lse, workspace, workspace_bytes=None, stream=None) -> None:
    """Enqueue one decode step (see ``oxd_paged_decode_run`` in include/oxd.h)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = lib().oxd_paged_decode_run(
        _handle(plan), _addr(q), _addr(k_pages), _addr(v_pages), _addr(indptr), _addr(indices),
        _addr(last_page_len), float(sm_scale), _addr(out), _addr(lse), _addr(workspace),
        int(workspace_bytes), _stream(stream, q))
    _check("oxd_paged_decode_run", st)


def oxd_plan_bind_workspace(plan, workspace, workspace_bytes=None, stream=None) -> None:
    """Enqueue the copy of the plan's work list into ``workspace``; later runs of
    the plan on that workspace copy nothing and launch with small parameter
    blocks (see ``oxd_plan_bind_workspace`` in include/oxd.h)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = lib().oxd_plan_bind_workspace(_handle(plan), _addr(workspace), int(workspace_bytes),
                                       _stream(stream, workspace))
    _check("oxd_plan_bind_workspace", st)


def oxd_paged_decode_run_static_workspace(plan, q, k_pages, v_pages, indptr, indices,
                                          last_page_len, sm_scale, out, lse,
                                          stream=None) -> None:
    """Enqueue one decode step using the library's own scratch array instead of a
    caller workspace (for callers that cannot allocate device memory; see
    ``oxd_paged_decode_run_static_workspace`` in include/oxd.h for its 32 MiB
    limit and the rule that overlapping calls race)."""
    st = lib().oxd_paged_decode_run_static_workspace(
        _handle(plan), _addr(q), _addr(k_pages), _addr(v_pages), _addr(indptr), _addr(indices),
        _addr(last_page_len), float(sm_scale), _addr(out), _addr(lse), _stream(stream, q))
    _check("oxd_paged_decode_run_static_workspace", st)


def oxd_read_static_workspace_status(stream=None) -> int:
    """Synchronise the stream and return the device status code of the last
    ``oxd_paged_decode_run_static_workspace`` call on the current device."""
    code = ctypes.c_int32()
    st = lib().oxd_read_static_workspace_status(_stream(stream), ctypes.byref(code))
    if st not in (OXD_OK, OXD_ERR_DEVICE_STATUS):
        _check("oxd_read_static_workspace_status", st)
    return code.value


def oxd_merge_states(v, s, N, S, H, D, v_out, s_out=None, stream=None) -> None:
    """Enqueue a state merge (see ``oxd_merge_states`` in include/oxd.h)."""
    st = lib().oxd_merge_states(_addr(v), _addr(s), int(N), int(S), int(H), int(D),
                                _addr(v_out), _addr(s_out), _stream(stream, v))
    _check("oxd_merge_states", st)


def oxd_plan_get_info(plan) -> PlanInfo:
    info = PlanInfo()
    _check("oxd_plan_get_info", lib().oxd_plan_get_info(_handle(plan), ctypes.byref(info)))
    return info


def oxd_plan_set_timing_events(plan, event_before, event_after) -> None:
    _check("oxd_plan_set_timing_events",
           lib().oxd_plan_set_timing_events(_handle(plan), _event(event_before),
                                            _event(event_after)))


def oxd_plan_destroy(plan) -> None:
    if isinstance(plan, Plan):
        plan.destroy()
    else:
        _check("oxd_plan_destroy", lib().oxd_plan_destroy(plan))


def oxd_read_device_status(workspace, stream=None) -> int:
    """Synchronise the stream and return the workspace's device status code."""
    code = ctypes.c_int32()
    st = lib().oxd_read_device_status(_addr(workspace), _stream(stream, workspace),
                                      ctypes.byref(code))
    if st not in (OXD_OK, OXD_ERR_DEVICE_STATUS):
        _check("oxd_read_device_status", st)
    return code.value


def make_desc(batch, num_qo_heads, num_kv_heads, page_size, layout, num_pages, head_dim=128,
              max_splits=0, force_splits=0, num_sms=0, tensor_path=0, shared_prefix_tokens=0,
              share_group=0, wait_timeout_ns=0, pdl=0) -> Desc:
    """Convenience constructor; ``layout`` may be "NHD"/"HND" or 0/1. A nonzero
    ``shared_prefix_tokens`` with ``share_group`` plans a cascade decode;
    ``wait_timeout_ns`` > 0 shortens the kernels' pipeline-wait limit;
    ``pdl`` = 1 launches a run's first kernel as a programmatic dependent of
    the kernel before it on the stream."""
    if isinstance(layout, str):
        layout = {"NHD": OXD_LAYOUT_NHD, "HND": OXD_LAYOUT_HND}[layout]
    return Desc(batch, num_qo_heads, num_kv_heads, head_dim, page_size, layout, num_pages,
                max_splits, force_splits, num_sms, tensor_path, shared_prefix_tokens,
                share_group, pdl, wait_timeout_ns)


def oxd_rope_append(desc: RopeAppendDesc, q, k, v, token_request, positions, indptr, indices,
                    page_refcount, q_out, k_pages, v_pages, workspace, workspace_bytes=None,
                    stream=None) -> None:
    """Enqueue a fused rotary embedding + paged KV append (see ``oxd_rope_append``
    in include/oxd.h)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = lib().oxd_rope_append(ctypes.byref(desc), _addr(q), _addr(k), _addr(v),
                               _addr(token_request), _addr(positions), _addr(indptr),
                               _addr(indices), _addr(page_refcount), _addr(q_out),
                               _addr(k_pages), _addr(v_pages), _addr(workspace),
                               int(workspace_bytes), _stream(stream, q))
    _check("oxd_rope_append", st)


# ------------------------------------------------------------------ causal prefill

class PrefillPlan:
    """Owns an ``oxd_prefill_plan`` handle (destroyed on :meth:`destroy` or garbage collection)."""

    def __init__(self, handle: int, workspace_bytes: int, desc: PrefillDesc):
        self.handle = handle
        self.workspace_bytes = workspace_bytes
        self.desc = desc

    @property
    def info(self) -> PrefillPlanInfo:
        return oxd_prefill_plan_get_info(self)

    def destroy(self):
        if self.handle:
            _check("oxd_prefill_plan_destroy", lib().oxd_prefill_plan_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            if self.handle:
                lib().oxd_prefill_plan_destroy(self.handle)
                self.handle = None
        except Exception:
            pass


def oxd_paged_prefill_plan(desc: PrefillDesc, qo_indptr_host, indptr_host, last_page_len_host,
                           device: int = 0) -> PrefillPlan:
    """Plan a causal prefill from host tables; returns a :class:`PrefillPlan`."""
    qo = np.ascontiguousarray(np.asarray(qo_indptr_host), dtype=np.int32)
    indptr = np.ascontiguousarray(np.asarray(indptr_host), dtype=np.int32)
    last = np.ascontiguousarray(np.asarray(last_page_len_host), dtype=np.int32)
    if (qo.shape != (desc.batch + 1,) or indptr.shape != (desc.batch + 1,)
            or last.shape != (desc.batch,)):
        raise OxdError("oxd_paged_prefill_plan", OXD_ERR_INVALID_ARGUMENT,
                       "qo_indptr and indptr must be [batch+1], last_page_len [batch]")
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    st = lib().oxd_paged_prefill_plan(ctypes.byref(desc), qo.ctypes.data, indptr.ctypes.data,
                                      last.ctypes.data, int(device), ctypes.byref(h),
                                      ctypes.byref(ws))
    _check("oxd_paged_prefill_plan", st)
    return PrefillPlan(h.value, ws.value, desc)


def oxd_paged_prefill_run(plan, q, k_pages, v_pages, qo_indptr, indptr, indices, last_page_len,
                          sm_scale, out, lse, workspace, workspace_bytes=None,
                          stream=None) -> None:
    """Enqueue one causal prefill (see ``oxd_paged_prefill_run`` in include/oxd.h)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = lib().oxd_paged_prefill_run(
        _handle(plan), _addr(q), _addr(k_pages), _addr(v_pages), _addr(qo_indptr),
        _addr(indptr), _addr(indices), _addr(last_page_len), float(sm_scale), _addr(out),
        _addr(lse), _addr(workspace), int(workspace_bytes), _stream(stream, q))
    _check("oxd_paged_prefill_run", st)


def oxd_prefill_plan_bind_workspace(plan, workspace, workspace_bytes=None, stream=None) -> None:
    """Enqueue the copy of the prefill plan's work list into ``workspace``."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    st = lib().oxd_prefill_plan_bind_workspace(_handle(plan), _addr(workspace),
                                               int(workspace_bytes), _stream(stream, workspace))
    _check("oxd_prefill_plan_bind_workspace", st)


def oxd_prefill_plan_get_info(plan) -> PrefillPlanInfo:
    info = PrefillPlanInfo()
    _check("oxd_prefill_plan_get_info",
           lib().oxd_prefill_plan_get_info(_handle(plan), ctypes.byref(info)))
    return info


def oxd_prefill_plan_set_timing_events(plan, event_before, event_after) -> None:
    _check("oxd_prefill_plan_set_timing_events",
           lib().oxd_prefill_plan_set_timing_events(_handle(plan), _event(event_before),
                                                    _event(event_after)))


def oxd_prefill_plan_destroy(plan) -> None:
    if isinstance(plan, PrefillPlan):
        plan.destroy()
    else:
        _check("oxd_prefill_plan_destroy", lib().oxd_prefill_plan_destroy(plan))
