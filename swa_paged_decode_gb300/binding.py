"""ctypes binding of libdsa_decode.so (include/dsa_decode.h).

Argument marshalling only: torch tensors become device pointers, strides and
sizes; every step of the decode runs in the library's CUDA kernels. The
functions keep the C names. Loading fails loudly when the library is missing
(there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import workloads as W

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libdsa_decode.so")

DSA_OK = 0
STATUS_NAMES = {0: "DSA_OK", -1: "DSA_ERR_INVALID_ARG", -2: "DSA_ERR_UNSUPPORTED",
                -3: "DSA_ERR_ALIGNMENT", -4: "DSA_ERR_WORKSPACE", -5: "DSA_ERR_CUDA",
                -6: "DSA_ERR_TIMEOUT", -7: "DSA_ERR_PLAN", -8: "DSA_ERR_BOUNDS"}
EXPORTED = ("dsa_decode_plan", "dsa_decode_plan_qk", "dsa_decode_run", "dsa_decode_combine", "dsa_decode_selection",
            "dsa_decode_read_status", "dsa_decode_status_string", "dsa_decode_abi_version",
            "dsa_decode_run_noalloc", "dsa_decode_run_v41", "dsa_decode_combine_v41")
DSA_ROPE_NEOX = 0
DSA_ROPE_GPTJ = 1


class DsaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} -> {STATUS_NAMES.get(status, status)}")
        self.status = status


class CacheDesc(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("num_pages", ctypes.c_int64),
                ("page_stride_bytes", ctypes.c_int64), ("page_size", ctypes.c_int32),
                ("format", ctypes.c_int32)]


class Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "magic", "abi_version", "num_tokens", "num_heads", "swa_width", "extra_width",
        "num_sms", "head_groups", "heads_per_group", "tiles_swa", "tiles_extra",
        "tiles_per_token", "units_per_cta", "ctas_per_group", "split_tokens", "kernel")] + \
        [(n, ctypes.c_int64) for n in (
            "total_units", "ws_sel_offset", "ws_part_lse_offset", "ws_part_sel_offset",
            "ws_part_o_offset", "workspace_bytes", "ws_bounds_offset", "balance_live",
            "ws_stage_offset", "workspace_bytes_mx", "wait_budget_cycles", "d_qk",
            "producer_q", "merge_in_run", "ws_count_offset")] + \
        [("reserved", ctypes.c_int64 * 7)]


_lib = None


class MxOutDesc(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("data_stride_t", ctypes.c_int64), ("data_stride_g", ctypes.c_int64),
                ("scale_stride_t", ctypes.c_int64), ("scale_stride_g", ctypes.c_int64),
                ("scale_stride_w", ctypes.c_int64), ("group_size", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class MxOut:
    """MXFP8 output buffers in the o-fused layout: data uint8 [T, H/G, G*512]
    (e4m3 codes), scale int32 [T, H/G, G*4] (ue8m0 bytes, four to a word)."""

    def __init__(self, T: int, H: int, group_size: int, device):
        assert H % group_size == 0
        G = group_size
        self.group_size = G
        self.data = torch.zeros((T, H // G, G * W.HEAD_DIM), dtype=torch.uint8, device=device)
        self.scale = torch.zeros((T, H // G, G * 4), dtype=torch.int32, device=device)

    def desc(self) -> MxOutDesc:
        d, s = self.data, self.scale
        return MxOutDesc(d.data_ptr(), s.data_ptr(), d.stride(0), d.stride(1), s.stride(0),
                         s.stride(1), s.stride(2), self.group_size, 0)

    def scale_bytes(self) -> torch.Tensor:
        """[T, H/G, G*16] uint8 (byte ka of a group's scales, little-endian words)."""
        return self.scale.contiguous().view(torch.uint8)


LIB_DEBUG_PATH = os.path.join(_HERE, "lib", "libdsa_decode_debug.so")
_libs = {}


def use_checking_build(on: bool):
    """Route every call of this module through the checking build
    (libdsa_decode_debug.so: bounds checks on every global and tile access,
    reported as DSA_ERR_BOUNDS) or back to the release library."""
    global _lib
    _lib = _load_path(LIB_DEBUG_PATH if on else LIB_PATH)
    return _lib


def load(path: str = LIB_PATH):
    """Load libdsa_decode.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = _load_path(path)
    return _lib


def _load_path(path: str):
    if path in _libs:
        return _libs[path]
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m swa_paged_decode_gb300.build`"
                           " (the CUDA library is required; there is no fallback)")
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.dsa_decode_plan.restype = ctypes.c_int
    lib.dsa_decode_plan.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(Plan),
                                    ctypes.POINTER(ctypes.c_size_t)]
    lib.dsa_decode_plan_qk.restype = ctypes.c_int
    lib.dsa_decode_plan_qk.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(Plan),
                                       ctypes.POINTER(ctypes.c_size_t)]
    lib.dsa_decode_run.restype = ctypes.c_int
    lib.dsa_decode_run.argtypes = [ctypes.POINTER(Plan), vp, ctypes.c_size_t, vp, i64, i64,
                                   ctypes.POINTER(CacheDesc), vp, i64, vp,
                                   ctypes.POINTER(CacheDesc), vp, i64, vp,
                                   vp, vp, vp, i64, ctypes.c_float, vp, vp, vp]
    lib.dsa_decode_combine.restype = ctypes.c_int
    lib.dsa_decode_combine.argtypes = [ctypes.POINTER(Plan), vp, ctypes.c_size_t, vp, vp, vp, vp]
    lib.dsa_decode_selection.restype = ctypes.c_int
    lib.dsa_decode_selection.argtypes = [ctypes.POINTER(Plan), vp, vp, vp, vp]
    lib.dsa_decode_read_status.restype = ctypes.c_int
    lib.dsa_decode_read_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32)]
    lib.dsa_decode_run_noalloc.restype = ctypes.c_int
    lib.dsa_decode_run_noalloc.argtypes = [ctypes.POINTER(Plan), vp, i64, i64,
                                           ctypes.POINTER(CacheDesc), vp, i64, vp,
                                           ctypes.POINTER(CacheDesc), vp, i64, vp,
                                           vp, vp, vp, i64, ctypes.c_float, vp, vp, vp, vp]
    lib.dsa_decode_run_v41.restype = ctypes.c_int
    lib.dsa_decode_run_v41.argtypes = [ctypes.POINTER(Plan), vp, ctypes.c_size_t, vp, i64, i64,
                                       ctypes.POINTER(CacheDesc), vp, i64, vp,
                                       ctypes.POINTER(CacheDesc), vp, i64, vp,
                                       vp, vp, vp, i64, i32, ctypes.c_float, vp,
                                       ctypes.POINTER(MxOutDesc), vp, vp]
    lib.dsa_decode_combine_v41.restype = ctypes.c_int
    lib.dsa_decode_combine_v41.argtypes = [ctypes.POINTER(Plan), vp, ctypes.c_size_t, vp, vp, vp,
                                           i64, i32, vp, ctypes.POINTER(MxOutDesc), vp, vp]
    lib.dsa_decode_status_string.restype = ctypes.c_char_p
    lib.dsa_decode_status_string.argtypes = [ctypes.c_int]
    lib.dsa_decode_abi_version.restype = ctypes.c_int32
    lib.dsa_decode_abi_version.argtypes = []
    _libs[path] = lib
    return lib


def _check(fn: str, rc: int):
    if rc != DSA_OK:
        raise DsaError(fn, rc)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def cache_desc(c: Optional[W.PagedCache]) -> Optional[CacheDesc]:
    if c is None:
        return None
    return CacheDesc(c.data.data_ptr(), c.num_pages, c.page_stride, c.page_size, c.fmt)


def dsa_decode_plan(num_tokens: int, num_heads: int, swa_width: int, extra_width: int = 0,
                    num_sms: int = 0):
    """-> (Plan, workspace_bytes)."""
    plan = Plan()
    ws = ctypes.c_size_t(0)
    _check("dsa_decode_plan", load().dsa_decode_plan(num_tokens, num_heads, swa_width,
                                                     extra_width, num_sms, ctypes.byref(plan),
                                                     ctypes.byref(ws)))
    return plan, int(ws.value)


def dsa_decode_plan_qk(num_tokens: int, num_heads: int, swa_width: int, extra_width: int = 0,
                       num_sms: int = 0, d_qk: int = 512):
    """-> (Plan, workspace_bytes) for key / query dims d_qk (512, or 576 for
    V3.2 records)."""
    plan = Plan()
    ws = ctypes.c_size_t(0)
    _check("dsa_decode_plan_qk", load().dsa_decode_plan_qk(num_tokens, num_heads, swa_width,
                                                           extra_width, num_sms, d_qk,
                                                           ctypes.byref(plan), ctypes.byref(ws)))
    return plan, int(ws.value)


def dsa_decode_run(plan: Plan, workspace: Optional[torch.Tensor], q: torch.Tensor,
                   swa_cache: W.PagedCache, swa_idx: torch.Tensor, swa_lens: torch.Tensor,
                   extra_cache: Optional[W.PagedCache], extra_idx: Optional[torch.Tensor],
                   extra_lens: Optional[torch.Tensor], sink: Optional[torch.Tensor],
                   positions: Optional[torch.Tensor], cos_sin: Optional[torch.Tensor],
                   scale: float, out: torch.Tensor, lse: torch.Tensor, stream=None,
                   check: bool = True) -> int:
    sc, ec = cache_desc(swa_cache), cache_desc(extra_cache)
    rc = load().dsa_decode_run(
        ctypes.byref(plan), _ptr(workspace), 0 if workspace is None else workspace.numel(),
        q.data_ptr(), q.stride(0), q.stride(1),
        ctypes.byref(sc), swa_idx.data_ptr(), swa_idx.stride(0), swa_lens.data_ptr(),
        None if ec is None else ctypes.byref(ec), _ptr(extra_idx),
        0 if extra_idx is None else extra_idx.stride(0), _ptr(extra_lens),
        _ptr(sink), _ptr(positions), _ptr(cos_sin),
        0 if cos_sin is None else cos_sin.shape[0], float(scale),
        out.data_ptr(), lse.data_ptr(), _stream(stream))
    if check:
        _check("dsa_decode_run", rc)
    return rc


def dsa_decode_combine(plan: Plan, workspace: Optional[torch.Tensor], sink: Optional[torch.Tensor],
                       out: torch.Tensor, lse: torch.Tensor, stream=None, check: bool = True) -> int:
    rc = load().dsa_decode_combine(ctypes.byref(plan), _ptr(workspace),
                                   0 if workspace is None else workspace.numel(), _ptr(sink),
                                   out.data_ptr(), lse.data_ptr(), _stream(stream))
    if check:
        _check("dsa_decode_combine", rc)
    return rc


def dsa_decode_run_v41(plan: Plan, workspace: Optional[torch.Tensor], q: torch.Tensor,
                       swa_cache: W.PagedCache, swa_idx: torch.Tensor, swa_lens: torch.Tensor,
                       extra_cache: Optional[W.PagedCache], extra_idx: Optional[torch.Tensor],
                       extra_lens: Optional[torch.Tensor], sink: Optional[torch.Tensor],
                       positions: Optional[torch.Tensor], cos_sin: Optional[torch.Tensor],
                       rope_style: int, scale: float, out: Optional[torch.Tensor],
                       mx: Optional[MxOut], lse: torch.Tensor, stream=None,
                       check: bool = True) -> int:
    sc, ec = cache_desc(swa_cache), cache_desc(extra_cache)
    md = None if mx is None else mx.desc()
    rc = load().dsa_decode_run_v41(
        ctypes.byref(plan), _ptr(workspace), 0 if workspace is None else workspace.numel(),
        q.data_ptr(), q.stride(0), q.stride(1),
        ctypes.byref(sc), swa_idx.data_ptr(), swa_idx.stride(0), swa_lens.data_ptr(),
        None if ec is None else ctypes.byref(ec), _ptr(extra_idx),
        0 if extra_idx is None else extra_idx.stride(0), _ptr(extra_lens),
        _ptr(sink), _ptr(positions), _ptr(cos_sin),
        0 if cos_sin is None else cos_sin.shape[0], int(rope_style), float(scale),
        _ptr(out), None if md is None else ctypes.byref(md), lse.data_ptr(), _stream(stream))
    if check:
        _check("dsa_decode_run_v41", rc)
    return rc


def dsa_decode_combine_v41(plan: Plan, workspace: Optional[torch.Tensor],
                           sink: Optional[torch.Tensor], positions: Optional[torch.Tensor],
                           cos_sin: Optional[torch.Tensor], rope_style: int,
                           out: Optional[torch.Tensor], mx: Optional[MxOut], lse: torch.Tensor,
                           stream=None, check: bool = True) -> int:
    md = None if mx is None else mx.desc()
    rc = load().dsa_decode_combine_v41(
        ctypes.byref(plan), _ptr(workspace), 0 if workspace is None else workspace.numel(),
        _ptr(sink), _ptr(positions), _ptr(cos_sin), 0 if cos_sin is None else cos_sin.shape[0],
        int(rope_style), _ptr(out), None if md is None else ctypes.byref(md), lse.data_ptr(),
        _stream(stream))
    if check:
        _check("dsa_decode_combine_v41", rc)
    return rc


def dsa_decode_selection(plan: Plan, workspace: torch.Tensor, kept: torch.Tensor,
                         checksum: torch.Tensor, stream=None):
    _check("dsa_decode_selection", load().dsa_decode_selection(
        ctypes.byref(plan), workspace.data_ptr(), kept.data_ptr(), checksum.data_ptr(),
        _stream(stream)))


def dsa_decode_read_status(workspace: torch.Tensor, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check("dsa_decode_read_status", load().dsa_decode_read_status(
        workspace.data_ptr(), _stream(stream), ctypes.byref(v)))
    return int(v.value)


def dsa_decode_run_noalloc(plan: Plan, q: torch.Tensor, swa_cache: W.PagedCache,
                           swa_idx: torch.Tensor, swa_lens: torch.Tensor,
                           extra_cache: Optional[W.PagedCache], extra_idx: Optional[torch.Tensor],
                           extra_lens: Optional[torch.Tensor], sink: Optional[torch.Tensor],
                           positions: Optional[torch.Tensor], cos_sin: Optional[torch.Tensor],
                           scale: float, out: torch.Tensor, lse: torch.Tensor,
                           device_status: Optional[torch.Tensor] = None, stream=None,
                           check: bool = True) -> int:
    """run + combine on the library's own device scratch (no workspace)."""
    sc, ec = cache_desc(swa_cache), cache_desc(extra_cache)
    rc = load().dsa_decode_run_noalloc(
        ctypes.byref(plan), q.data_ptr(), q.stride(0), q.stride(1),
        ctypes.byref(sc), swa_idx.data_ptr(), swa_idx.stride(0), swa_lens.data_ptr(),
        None if ec is None else ctypes.byref(ec), _ptr(extra_idx),
        0 if extra_idx is None else extra_idx.stride(0), _ptr(extra_lens),
        _ptr(sink), _ptr(positions), _ptr(cos_sin),
        0 if cos_sin is None else cos_sin.shape[0], float(scale),
        out.data_ptr(), lse.data_ptr(), _ptr(device_status), _stream(stream))
    if check:
        _check("dsa_decode_run_noalloc", rc)
    return rc


class Decoder:
    """Plan + workspace for one workload shape; ``__call__`` runs run+combine
    on the current stream. Allocation uses torch; compute is the library's.
    With ``mx_group`` the output is MXFP8 (``self.mx``, o-fused with that many
    heads per group) instead of bf16 ``self.out``; a GPT-J workload or an
    MXFP8 output goes through the V4.1 entry points."""

    def __init__(self, w: W.Workload, num_sms: int = 0, mx_group: Optional[int] = None):
        self.plan, nbytes = dsa_decode_plan_qk(w.T, w.H, w.swa.width,
                                               0 if w.extra is None else w.extra.width, num_sms,
                                               int(w.q.shape[-1]))
        dev = w.q.device
        if mx_group is not None:
            nbytes = self.plan.workspace_bytes_mx
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        self.mx = None if mx_group is None else MxOut(w.T, w.H, mx_group, dev)
        self.out = (torch.empty((w.T, w.H, W.HEAD_DIM), dtype=torch.bfloat16, device=dev)
                    if self.mx is None else None)
        self.lse = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)

    def __call__(self, w: W.Workload, stream=None):
        ei = None if w.extra is None else w.extra.ids
        el = None if w.extra is None else w.extra.lens
        if self.mx is None and w.rope_style == DSA_ROPE_NEOX:
            dsa_decode_run(self.plan, self.workspace, w.q, w.swa_cache, w.swa.ids, w.swa.lens,
                           w.extra_cache, ei, el, w.sink, w.positions, w.cos_sin, w.scale,
                           self.out, self.lse, stream)
            dsa_decode_combine(self.plan, self.workspace, w.sink, self.out, self.lse, stream)
            return self.out, self.lse
        dsa_decode_run_v41(self.plan, self.workspace, w.q, w.swa_cache, w.swa.ids, w.swa.lens,
                           w.extra_cache, ei, el, w.sink, w.positions, w.cos_sin, w.rope_style,
                           w.scale, self.out, self.mx, self.lse, stream)
        dsa_decode_combine_v41(self.plan, self.workspace, w.sink, w.positions, w.cos_sin,
                               w.rope_style, self.out, self.mx, self.lse, stream)
        return (self.out if self.mx is None else self.mx), self.lse

    def selection(self, stream=None):
        dev = self.lse.device
        kept = torch.empty(self.plan.num_tokens, dtype=torch.int32, device=dev)
        chk = torch.empty(self.plan.num_tokens, dtype=torch.int32, device=dev)
        dsa_decode_selection(self.plan, self.workspace, kept, chk, stream)
        return kept, chk
