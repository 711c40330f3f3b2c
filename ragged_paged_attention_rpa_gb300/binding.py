"""Thin ctypes binding of librpa (include/rpa.h): argument marshalling only.

Every computation runs in the library's CUDA kernels; this module turns torch
tensors and numpy arrays into pointers and sizes, and status codes into
exceptions.  It never falls back to another implementation: if librpa.so is
missing or fails to load, every call raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "librpa.so")

RPA_OK = 0
RPA_ERR_INVALID_ARG = -1
RPA_ERR_UNSUPPORTED = -2
RPA_ERR_WORKSPACE_TOO_SMALL = -3
RPA_ERR_CUDA = -4
RPA_ERR_DEVICE = -5
RPA_ERR_PLAN_MISMATCH = -6

RPA_DTYPE_BF16 = 0
RPA_DTYPE_F32 = 1
RPA_DTYPE_FP8_E4M3 = 2

RPA_DEVERR_NONE = 0
RPA_DEVERR_PAGE_ID = 1
RPA_DEVERR_LENGTHS = 2
RPA_DEVERR_PLAN = 3
RPA_DEVERR_TIMEOUT = 4

RPA_PATH_AUTO = 0
RPA_PATH_SIMT = 1
RPA_PATH_TC = 2

EXPORTS = ["rpa_plan", "rpa_plan_destroy", "rpa_plan_get_info", "rpa_forward",
           "rpa_get_device_error", "rpa_clear_device_error", "rpa_trace_begin",
           "rpa_trace_end", "rpa_status_string", "rpa_forward_decode_noalloc",
           "rpa_write_kv", "rpa_forward_kv", "rpa_forward_fp8kv", "rpa_qkv_prologue",
           "rpa_forward_qkv", "rpa_last_cuda_error"]

RPA_KERNEL_NAMES = {0: "decode_split", 1: "decode_combine", 2: "prefill_tc", 3: "simt",
                    4: "kv_write", 5: "prologue", 6: "prefill_combine"}


class QkvNorm(ctypes.Structure):
    """rpa_qkv_norm: norm weights (device float32 [head_dim] or None), eps and
    the rotary base (<= 0: no rotation)."""
    _fields_ = [("q_weight", ctypes.c_void_p), ("k_weight", ctypes.c_void_p),
                ("v_weight", ctypes.c_void_p), ("eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float)]


class RpaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        self.cuda_error = 0
        msg = "%s: %s" % (where, status_string(status))
        if status == RPA_ERR_CUDA:
            try:
                self.cuda_error = int(lib().rpa_last_cuda_error())
                msg += " (cudaError %d)" % self.cuda_error
            except Exception:  # noqa: BLE001 - diagnostics only
                pass
        super().__init__(msg)


class _Options(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_int32), ("path", ctypes.c_int32),
                ("q_block", ctypes.c_int32), ("kv_split", ctypes.c_int32),
                ("num_sms", ctypes.c_int32), ("prefill_pairs", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("prefill_split", ctypes.c_int32),
                ("decode_sms", ctypes.c_int32), ("decode_kernel", ctypes.c_int32),
                ("prefill_dynamic", ctypes.c_int32), ("prefill_grouping", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("num_decode_seqs", ctypes.c_int32),
                ("num_prefill_seqs", ctypes.c_int32), ("q_block", ctypes.c_int32),
                ("kv_split", ctypes.c_int32), ("max_splits", ctypes.c_int32),
                ("num_prefill_items", ctypes.c_int32), ("prefill_ctas", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64), ("prefill_pairs", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("prefill_split_items", ctypes.c_int32),
                ("prefill_split_parts", ctypes.c_int32), ("prefill_max_tiles", ctypes.c_int32),
                ("decode_sms", ctypes.c_int32), ("prefill_sms", ctypes.c_int32),
                ("decode_kernel", ctypes.c_int32), ("prefill_dynamic", ctypes.c_int32),
                ("prefill_groups", ctypes.c_int32)]

    def as_dict(self):
        return {name: int(getattr(self, name)) for name, _ in self._fields_}


class _TraceRecord(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("ms", ctypes.c_float)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load librpa.so from the package directory (built by ``build.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "librpa.so is not built (%s); run "
                "`python -m ragged_paged_attention_rpa_gb300.build`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        i32, vp, sz = ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
        L.rpa_plan.argtypes = [ctypes.POINTER(vp), vp, vp, vp, i32, i32, i32, i32, i32, i32,
                               i32, i32, ctypes.POINTER(_Options), ctypes.POINTER(sz)]
        L.rpa_plan.restype = i32
        L.rpa_plan_destroy.argtypes = [vp]
        L.rpa_plan_destroy.restype = i32
        L.rpa_plan_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
        L.rpa_plan_get_info.restype = i32
        L.rpa_forward.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp,
                                  ctypes.c_float, vp, vp, vp, vp, sz]
        L.rpa_forward.restype = i32
        L.rpa_forward_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                  i32, vp, ctypes.c_float, vp, vp, vp]
        L.rpa_forward_decode_noalloc.restype = i32
        L.rpa_write_kv.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                   i32, vp, vp]
        L.rpa_write_kv.restype = i32
        L.rpa_forward_kv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp,
                                     ctypes.c_float, vp, vp, vp, vp, ctypes.c_size_t]
        L.rpa_forward_kv.restype = i32
        L.rpa_forward_fp8kv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                        vp, ctypes.c_float, vp, vp, vp, vp, ctypes.c_size_t]
        L.rpa_forward_fp8kv.restype = i32
        L.rpa_qkv_prologue.argtypes = [vp, vp, vp, ctypes.POINTER(QkvNorm), vp, vp, vp, vp, vp,
                                       vp, i32, i32, i32, i32, i32, i32, i32, i32, i32, vp, vp]
        L.rpa_qkv_prologue.restype = i32
        L.rpa_forward_qkv.argtypes = [vp, vp, vp, ctypes.POINTER(QkvNorm), vp, vp, vp, vp, vp,
                                      vp, i32, i32, i32, i32, i32, vp, ctypes.c_float, vp, vp,
                                      vp, vp, ctypes.c_size_t]
        L.rpa_forward_qkv.restype = i32
        L.rpa_get_device_error.argtypes = [vp, vp, ctypes.POINTER(i32)]
        L.rpa_get_device_error.restype = i32
        L.rpa_clear_device_error.argtypes = [vp, vp]
        L.rpa_clear_device_error.restype = i32
        L.rpa_trace_begin.argtypes = [i32]
        L.rpa_trace_begin.restype = i32
        L.rpa_trace_end.argtypes = [ctypes.POINTER(_TraceRecord), ctypes.POINTER(i32)]
        L.rpa_trace_end.restype = i32
        L.rpa_last_cuda_error.argtypes = []
        L.rpa_last_cuda_error.restype = i32
        L.rpa_status_string.argtypes = [i32]
        L.rpa_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().rpa_status_string(int(status)).decode()


def _np_i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def _np_ptr(a):
    # The address as an int (ctypes passes it as void*): data_as() costs
    # ~2 us a call, a third of this binding's per-plan overhead.
    return None if a is None else a.ctypes.data


class Plan:
    """A librpa plan (rpa_plan); freed with rpa_plan_destroy when collected."""

    def __init__(self, handle, workspace_bytes: int, meta: dict):
        self._handle = handle
        self.workspace_bytes = int(workspace_bytes)
        self.meta = meta

    @property
    def handle(self):
        if self._handle is None:
            raise RuntimeError("plan already destroyed")
        return self._handle

    def info(self) -> dict:
        inf = PlanInfo()
        st = lib().rpa_plan_get_info(self.handle, ctypes.byref(inf))
        if st != RPA_OK:
            raise RpaError(st, "rpa_plan_get_info")
        return inf.as_dict()

    def destroy(self):
        if self._handle is not None and _lib is not None:
            _lib.rpa_plan_destroy(self._handle)
        self._handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def rpa_plan(cu_q_lens_host, kv_lens_host, window_host, num_q_heads: int,
             num_kv_heads: int, head_dim: int, page_size: int, max_pages_per_seq: int,
             num_pages: int, dtype: int = RPA_DTYPE_BF16, path: int = RPA_PATH_AUTO,
             q_block: int = 0, kv_split: int = 0, num_sms: int = 0,
             prefill_pairs: int = 0, kv_dtype: int = 0, prefill_split: int = 0,
             decode_sms: int = 0, decode_kernel: int = 0,
             prefill_dynamic: int = 0, prefill_grouping: int = 0) -> Plan:
    """rpa_plan from host (numpy) metadata; returns a Plan."""
    cu = _np_i32(cu_q_lens_host)
    kv = _np_i32(kv_lens_host)
    win = _np_i32(window_host)
    num_seqs = int(kv.shape[0])
    if cu.shape[0] != num_seqs + 1:
        raise ValueError("cu_q_lens must have num_seqs + 1 entries")
    if win is not None and win.shape[0] != num_seqs:
        raise ValueError("window must have num_seqs entries")
    opts = _Options(ctypes.sizeof(_Options), path, q_block, kv_split, num_sms, prefill_pairs,
                    kv_dtype, prefill_split, decode_sms, decode_kernel, prefill_dynamic,
                    prefill_grouping)
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    st = lib().rpa_plan(ctypes.byref(handle), _np_ptr(cu), _np_ptr(kv), _np_ptr(win),
                        num_seqs, num_q_heads, num_kv_heads, head_dim, page_size,
                        max_pages_per_seq, num_pages, dtype, ctypes.byref(opts),
                        ctypes.byref(ws))
    if st != RPA_OK:
        raise RpaError(st, "rpa_plan")
    meta = dict(num_seqs=num_seqs, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                head_dim=head_dim, page_size=page_size, has_window=win is not None,
                dtype=dtype, total_q=int(cu[-1]))
    return Plan(handle.value, ws.value, meta)


def _dptr(t, name, dtype=None):
    import torch
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t.data_ptr()


def _stream_ptr(stream):
    import torch
    if stream is None:
        # The current stream's handle without building a Stream object.
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return raw(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def rpa_forward(q, k_pages, v_pages, page_table, cu_q_lens, kv_lens, window,
                sm_scale: float, out, plan: Plan, workspace, stream=None) -> None:
    """rpa_forward on torch CUDA tensors; enqueues on `stream` (default: current)."""
    import torch
    m = plan.meta
    dt = torch.bfloat16 if m["dtype"] == RPA_DTYPE_BF16 else torch.float32
    st = lib().rpa_forward(
        _dptr(q, "q", dt), _dptr(k_pages, "k_pages", dt), _dptr(v_pages, "v_pages", dt),
        _dptr(page_table, "page_table", torch.int32), _dptr(cu_q_lens, "cu_q_lens", torch.int32),
        _dptr(kv_lens, "kv_lens", torch.int32), m["num_seqs"], m["num_q_heads"],
        m["num_kv_heads"], m["head_dim"], m["page_size"],
        _dptr(window, "window", torch.int32), float(sm_scale), _dptr(out, "out", dt),
        _stream_ptr(stream), plan.handle, _dptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size())
    if st != RPA_OK:
        raise RpaError(st, "rpa_forward")


def rpa_write_kv(k_new, v_new, k_pages, v_pages, page_table, cu_q_lens, kv_lens,
                 num_pages: int, workspace=None, stream=None) -> None:
    """rpa_write_kv on torch CUDA tensors: scatter the new tokens' K/V rows
    ([total_q, Hkv, D]) into their pages."""
    import torch
    dt = k_pages.dtype
    dtype = RPA_DTYPE_BF16 if dt == torch.bfloat16 else RPA_DTYPE_F32
    total_q, hkv, d = (int(x) for x in k_new.shape)
    st = lib().rpa_write_kv(
        _dptr(k_new, "k_new", dt), _dptr(v_new, "v_new", dt), _dptr(k_pages, "k_pages", dt),
        _dptr(v_pages, "v_pages", dt), _dptr(page_table, "page_table", torch.int32),
        _dptr(cu_q_lens, "cu_q_lens", torch.int32), _dptr(kv_lens, "kv_lens", torch.int32),
        int(kv_lens.numel()), total_q, hkv, d, int(k_pages.shape[1]), int(page_table.shape[1]),
        int(num_pages), dtype, _dptr(workspace, "workspace"), _stream_ptr(stream))
    if st != RPA_OK:
        raise RpaError(st, "rpa_write_kv")


def qkv_norm(q_weight=None, k_weight=None, v_weight=None, eps: float = 1e-6,
             rope_theta: float = 10000.0) -> QkvNorm:
    """An rpa_qkv_norm over device float32 weight tensors (kept alive by the
    caller)."""
    import torch
    return QkvNorm(_dptr(q_weight, "q_weight", torch.float32),
                   _dptr(k_weight, "k_weight", torch.float32),
                   _dptr(v_weight, "v_weight", torch.float32), float(eps), float(rope_theta))


def rpa_qkv_prologue(q, k, v, norm: QkvNorm, q_out, k_pages, v_pages, page_table, cu_q_lens,
                     kv_lens, num_pages: int, workspace=None, stream=None) -> None:
    """rpa_qkv_prologue on torch CUDA tensors: q/k RMS norm + rotary embedding,
    v norm; q to q_out, k and v rows into their pages."""
    import torch
    dt = q.dtype
    dtype = RPA_DTYPE_BF16 if dt == torch.bfloat16 else RPA_DTYPE_F32
    total_q, hq, d = (int(x) for x in q.shape)
    hkv = int(k.shape[1])
    st = lib().rpa_qkv_prologue(
        _dptr(q, "q", dt), _dptr(k, "k", dt), _dptr(v, "v", dt), ctypes.byref(norm),
        _dptr(q_out, "q_out", dt), _dptr(k_pages, "k_pages", dt), _dptr(v_pages, "v_pages", dt),
        _dptr(page_table, "page_table", torch.int32),
        _dptr(cu_q_lens, "cu_q_lens", torch.int32), _dptr(kv_lens, "kv_lens", torch.int32),
        int(kv_lens.numel()), total_q, hq, hkv, d, int(k_pages.shape[1]),
        int(page_table.shape[1]), int(num_pages), dtype, _dptr(workspace, "workspace"),
        _stream_ptr(stream))
    if st != RPA_OK:
        raise RpaError(st, "rpa_qkv_prologue")


def rpa_forward_qkv(q, k, v, norm: QkvNorm, q_buf, k_pages, v_pages, page_table, cu_q_lens,
                    kv_lens, window, sm_scale: float, out, plan: "Plan", workspace,
                    stream=None) -> None:
    """rpa_forward_qkv: the prologue into q_buf and the pages, then attention."""
    ForwardQkvCall(q, k, v, norm, q_buf, k_pages, v_pages, page_table, cu_q_lens, kv_lens,
                   window, sm_scale, out, plan, workspace, stream)()


def rpa_forward_fp8kv(q, k_pages, v_pages, k_scale, v_scale, page_table, cu_q_lens, kv_lens,
                      window, sm_scale: float, out, plan: Plan, workspace, stream=None) -> None:
    """rpa_forward_fp8kv: decode over e4m3 K/V pages (uint8 tensors) with
    float32 per-KV-head scales."""
    import torch
    m = plan.meta
    st = lib().rpa_forward_fp8kv(
        _dptr(q, "q", torch.bfloat16), _dptr(k_pages, "k_pages", torch.uint8),
        _dptr(v_pages, "v_pages", torch.uint8), _dptr(k_scale, "k_scale", torch.float32),
        _dptr(v_scale, "v_scale", torch.float32),
        _dptr(page_table, "page_table", torch.int32), _dptr(cu_q_lens, "cu_q_lens", torch.int32),
        _dptr(kv_lens, "kv_lens", torch.int32), m["num_seqs"], m["num_q_heads"],
        m["num_kv_heads"], m["head_dim"], m["page_size"],
        _dptr(window, "window", torch.int32), float(sm_scale), _dptr(out, "out", torch.bfloat16),
        _stream_ptr(stream), plan.handle, _dptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size())
    if st != RPA_OK:
        raise RpaError(st, "rpa_forward_fp8kv")


def rpa_forward_kv(q, k_new, v_new, k_pages, v_pages, page_table, cu_q_lens, kv_lens, window,
                   sm_scale: float, out, plan: Plan, workspace, stream=None) -> None:
    """rpa_forward_kv: write the new tokens' K/V into their pages, then attend."""
    import torch
    m = plan.meta
    dt = torch.bfloat16 if m["dtype"] == RPA_DTYPE_BF16 else torch.float32
    st = lib().rpa_forward_kv(
        _dptr(q, "q", dt), _dptr(k_new, "k_new", dt), _dptr(v_new, "v_new", dt),
        _dptr(k_pages, "k_pages", dt), _dptr(v_pages, "v_pages", dt),
        _dptr(page_table, "page_table", torch.int32), _dptr(cu_q_lens, "cu_q_lens", torch.int32),
        _dptr(kv_lens, "kv_lens", torch.int32), m["num_seqs"], m["num_q_heads"],
        m["num_kv_heads"], m["head_dim"], m["page_size"],
        _dptr(window, "window", torch.int32), float(sm_scale), _dptr(out, "out", dt),
        _stream_ptr(stream), plan.handle, _dptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size())
    if st != RPA_OK:
        raise RpaError(st, "rpa_forward_kv")


def rpa_forward_decode_noalloc(q, k_pages, v_pages, page_table, cu_q_lens, kv_lens, window,
                               sm_scale: float, out, plan: Plan, stream=None) -> None:
    """rpa_forward_decode_noalloc: decode with the library's fixed scratch
    array instead of a caller workspace (see include/rpa.h)."""
    import torch
    m = plan.meta
    dt = torch.bfloat16
    st = lib().rpa_forward_decode_noalloc(
        _dptr(q, "q", dt), _dptr(k_pages, "k_pages", dt), _dptr(v_pages, "v_pages", dt),
        _dptr(page_table, "page_table", torch.int32), _dptr(cu_q_lens, "cu_q_lens", torch.int32),
        _dptr(kv_lens, "kv_lens", torch.int32), m["num_seqs"], m["num_q_heads"],
        m["num_kv_heads"], m["head_dim"], m["page_size"],
        _dptr(window, "window", torch.int32), float(sm_scale), _dptr(out, "out", dt),
        _stream_ptr(stream), plan.handle)
    if st != RPA_OK:
        raise RpaError(st, "rpa_forward_decode_noalloc")


def rpa_get_device_error(workspace, stream=None) -> int:
    """Read and clear the device error word (synchronises the stream)."""
    err = ctypes.c_int32(0)
    st = lib().rpa_get_device_error(_dptr(workspace, "workspace"), _stream_ptr(stream),
                                    ctypes.byref(err))
    if st not in (RPA_OK, RPA_ERR_DEVICE):
        raise RpaError(st, "rpa_get_device_error")
    return int(err.value)


def rpa_clear_device_error(workspace, stream=None) -> None:
    st = lib().rpa_clear_device_error(_dptr(workspace, "workspace"), _stream_ptr(stream))
    if st != RPA_OK:
        raise RpaError(st, "rpa_clear_device_error")


def rpa_trace_begin(capacity: int) -> None:
    st = lib().rpa_trace_begin(int(capacity))
    if st != RPA_OK:
        raise RpaError(st, "rpa_trace_begin")


def rpa_trace_end(max_records: int = 65536):
    """Stop tracing; returns [(kernel name, device ms), ...] in launch order."""
    recs = (_TraceRecord * max_records)()
    n = ctypes.c_int32(max_records)
    st = lib().rpa_trace_end(recs, ctypes.byref(n))
    if st != RPA_OK:
        raise RpaError(st, "rpa_trace_end")
    return [(RPA_KERNEL_NAMES.get(recs[i].kernel, str(recs[i].kernel)), float(recs[i].ms))
            for i in range(n.value)]


def rpa_status_string(status: int) -> str:
    return status_string(status)


def alloc_workspace(plan: Plan, device=None):
    """A workspace tensor of the plan's size (caller-owned; 256-B aligned)."""
    import torch
    n = max(256, plan.workspace_bytes)
    ws = torch.zeros(n, dtype=torch.uint8, device=device or "cuda")
    assert ws.data_ptr() % 256 == 0
    return ws


class Batch:
    """Device copies of a workloads.Batch, ready for rpa_forward."""

    def __init__(self, b, device="cuda", stream=None):
        import torch
        self.src = b
        dt = torch.bfloat16 if b.dtype == "bf16" else torch.float32

        def dev(a, dtype):
            t = torch.from_numpy(np.ascontiguousarray(a))
            if dtype is torch.bfloat16:
                t = t.view(torch.int16).view(torch.bfloat16)
            return t.to(device, non_blocking=False)

        self.q = dev(b.q, dt)
        self.k_pages = dev(b.k_pages, dt)
        self.v_pages = dev(b.v_pages, dt)
        self.page_table = dev(b.page_table, torch.int32)
        self.cu_q_lens = dev(b.cu_q_lens, torch.int32)
        self.kv_lens = dev(b.kv_lens, torch.int32)
        self.window = None if b.window is None else dev(b.window, torch.int32)
        self.out = torch.empty_like(self.q)
        self.dtype = RPA_DTYPE_BF16 if b.dtype == "bf16" else RPA_DTYPE_F32

    def plan(self, **kw) -> Plan:
        b = self.src
        return rpa_plan(b.cu_q_lens, b.kv_lens, b.window, b.num_q_heads, b.num_kv_heads,
                        b.head_dim, b.page_size, b.max_pages_per_seq, b.num_pages,
                        dtype=self.dtype, **kw)

    def call(self, plan: Plan, workspace, stream=None) -> "ForwardCall":
        return ForwardCall(self.q, self.k_pages, self.v_pages, self.page_table,
                           self.cu_q_lens, self.kv_lens, self.window, self.src.sm_scale,
                           self.out, plan, workspace, stream)

    def forward(self, plan: Plan, workspace, stream=None, out=None):
        rpa_forward(self.q, self.k_pages, self.v_pages, self.page_table, self.cu_q_lens,
                    self.kv_lens, self.window, self.src.sm_scale,
                    self.out if out is None else out, plan, workspace, stream)
        return self.out if out is None else out


class ForwardCall:
    """rpa_forward with its arguments marshalled once (for tight launch loops).

    Holds references to every tensor it points at; calling it enqueues one
    rpa_forward on the stream given at construction (default: current).
    """

    def __init__(self, q, k_pages, v_pages, page_table, cu_q_lens, kv_lens, window,
                 sm_scale: float, out, plan: Plan, workspace, stream=None):
        import torch
        m = plan.meta
        dt = torch.bfloat16 if m["dtype"] == RPA_DTYPE_BF16 else torch.float32
        self._keep = (q, k_pages, v_pages, page_table, cu_q_lens, kv_lens, window, out,
                      plan, workspace)
        self._args = (
            _dptr(q, "q", dt), _dptr(k_pages, "k_pages", dt), _dptr(v_pages, "v_pages", dt),
            _dptr(page_table, "page_table", torch.int32),
            _dptr(cu_q_lens, "cu_q_lens", torch.int32),
            _dptr(kv_lens, "kv_lens", torch.int32), m["num_seqs"], m["num_q_heads"],
            m["num_kv_heads"], m["head_dim"], m["page_size"],
            _dptr(window, "window", torch.int32), float(sm_scale), _dptr(out, "out", dt),
            _stream_ptr(stream), plan.handle, _dptr(workspace, "workspace"),
            workspace.numel() * workspace.element_size())
        self._fn = lib().rpa_forward

    def __call__(self, plan: Optional[Plan] = None):
        """Enqueue the call; `plan` replaces the plan given at construction
        (one built for the same metadata, e.g. anew for every step)."""
        args = self._args
        if plan is not None:
            args = args[:15] + (plan.handle,) + args[16:]
        st = self._fn(*args)
        if st != RPA_OK:
            raise RpaError(st, "rpa_forward")


class ForwardFp8Call(ForwardCall):
    """rpa_forward_fp8kv (decode over e4m3 pages) with its arguments
    marshalled once."""

    def __init__(self, q, k_fp8, v_fp8, k_scale, v_scale, page_table, cu_q_lens, kv_lens,
                 window, sm_scale: float, out, plan: Plan, workspace, stream=None):
        import torch
        m = plan.meta
        self._keep = (q, k_fp8, v_fp8, k_scale, v_scale, page_table, cu_q_lens, kv_lens, window,
                      out, plan, workspace)
        self._args = (
            _dptr(q, "q", torch.bfloat16), _dptr(k_fp8, "k_pages", torch.uint8),
            _dptr(v_fp8, "v_pages", torch.uint8), _dptr(k_scale, "k_scale", torch.float32),
            _dptr(v_scale, "v_scale", torch.float32),
            _dptr(page_table, "page_table", torch.int32),
            _dptr(cu_q_lens, "cu_q_lens", torch.int32),
            _dptr(kv_lens, "kv_lens", torch.int32), m["num_seqs"], m["num_q_heads"],
            m["num_kv_heads"], m["head_dim"], m["page_size"],
            _dptr(window, "window", torch.int32), float(sm_scale),
            _dptr(out, "out", torch.bfloat16), _stream_ptr(stream), plan.handle,
            _dptr(workspace, "workspace"), workspace.numel() * workspace.element_size())
        self._fn = lib().rpa_forward_fp8kv

    def __call__(self, plan: Optional[Plan] = None):
        args = self._args
        if plan is not None:
            args = args[:17] + (plan.handle,) + args[18:]
        st = self._fn(*args)
        if st != RPA_OK:
            raise RpaError(st, "rpa_forward_fp8kv")


class ForwardKvCall(ForwardCall):
    """rpa_forward_kv (write the new tokens' K/V, then attend) with its
    arguments marshalled once."""

    def __init__(self, q, k_new, v_new, k_pages, v_pages, page_table, cu_q_lens, kv_lens,
                 window, sm_scale: float, out, plan: Plan, workspace, stream=None):
        import torch
        super().__init__(q, k_pages, v_pages, page_table, cu_q_lens, kv_lens, window,
                         sm_scale, out, plan, workspace, stream)
        dt = torch.bfloat16 if plan.meta["dtype"] == RPA_DTYPE_BF16 else torch.float32
        self._keep = self._keep + (k_new, v_new)
        a = self._args
        self._args = (a[0], _dptr(k_new, "k_new", dt), _dptr(v_new, "v_new", dt)) + a[1:]
        self._fn = lib().rpa_forward_kv

    def __call__(self):
        st = self._fn(*self._args)
        if st != RPA_OK:
            raise RpaError(st, "rpa_forward_kv")


class ForwardQkvCall(ForwardCall):
    """rpa_forward_qkv (q/k/v prologue, then attention) with its arguments
    marshalled once."""

    def __init__(self, q, k, v, norm: QkvNorm, q_buf, k_pages, v_pages, page_table, cu_q_lens,
                 kv_lens, window, sm_scale: float, out, plan: "Plan", workspace, stream=None):
        import torch
        m = plan.meta
        dt = torch.bfloat16 if m["dtype"] == RPA_DTYPE_BF16 else torch.float32
        self._norm = norm
        self._keep = (q, k, v, q_buf, k_pages, v_pages, page_table, cu_q_lens, kv_lens, window,
                      out, plan, workspace)
        self._args = (
            _dptr(q, "q", dt), _dptr(k, "k", dt), _dptr(v, "v", dt), ctypes.byref(norm),
            _dptr(q_buf, "q_buf", dt), _dptr(k_pages, "k_pages", dt),
            _dptr(v_pages, "v_pages", dt), _dptr(page_table, "page_table", torch.int32),
            _dptr(cu_q_lens, "cu_q_lens", torch.int32),
            _dptr(kv_lens, "kv_lens", torch.int32), m["num_seqs"], m["num_q_heads"],
            m["num_kv_heads"], m["head_dim"], m["page_size"],
            _dptr(window, "window", torch.int32), float(sm_scale), _dptr(out, "out", dt),
            _stream_ptr(stream), plan.handle, _dptr(workspace, "workspace"),
            workspace.numel() * workspace.element_size())
        self._fn = lib().rpa_forward_qkv

    def __call__(self):
        st = self._fn(*self._args)
        if st != RPA_OK:
            raise RpaError(st, "rpa_forward_qkv")
