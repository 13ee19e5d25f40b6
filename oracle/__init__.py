"""fp64 CPU oracle for paged sparse/sliding-window MQA decode attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use this package. The product library never
imports it, and it imports nothing from the product package.

``dsa_oracle.c`` holds the definition (candidate rows, record dequantization,
NeoX or GPT-J RoPE of Q, scores, lse and the sink-weighted output; the V4.1
output epilogue: inverse RoPE, MXFP8 cast, o-fused layout). This module only
compiles it with gcc, marshals numpy/torch CPU arrays into it, and adds
``combine`` -- the split-KV merge written as the plain formula from the
"production.py" page's Python KV merge (out = sum_i e^{lse_i} O_i /
sum_i e^{lse_i}) extended by the sink term of the vLLM swapab page's merge
step (the denominator gains e^{sink}).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

FMT_FP8_528 = 0
FMT_NVFP4_288 = 1
FMT_FP8_528_UE8M0 = 2
FMT_MODEL1_584 = 3
FMT_V32_656 = 4
RECORD_BYTES = {FMT_FP8_528: 528, FMT_NVFP4_288: 288, FMT_FP8_528_UE8M0: 528, FMT_MODEL1_584: 584,
                FMT_V32_656: 656}
KEY_DIMS = {FMT_V32_656: 576}   # formats whose keys have more than 512 dims
ROPE_NEOX = 0
ROPE_GPTJ = 1


def build(force: bool = False) -> str:
    """Compile dsa_oracle.c into liboracle.so next to it (gcc, -O2, no fast-math,
    no contraction of products and sums into fused multiply-adds)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-Wall", "-ffp-contract=off",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class _Cache(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("num_pages", ctypes.c_int64),
                ("page_stride", ctypes.c_int64), ("page_size", ctypes.c_int32),
                ("format", ctypes.c_int32)]


class _List(ctypes.Structure):
    _fields_ = [("ids", ctypes.c_void_p), ("lens", ctypes.c_void_p),
                ("row_stride", ctypes.c_int64), ("width", ctypes.c_int32),
                ("pad_", ctypes.c_int32)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_e4m3_value.restype = ctypes.c_double
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_value.restype = ctypes.c_double
            lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
            lib.oracle_dequant_record.restype = None
            lib.oracle_dequant_record.argtypes = [ctypes.c_void_p, ctypes.c_int32,
                                                  ctypes.c_void_p]
            lib.oracle_ue8m0_value.restype = ctypes.c_double
            lib.oracle_ue8m0_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
            lib.oracle_ue8m0_ceil.restype = ctypes.c_uint8
            lib.oracle_ue8m0_ceil.argtypes = [ctypes.c_float]
            lib.oracle_decode.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [
                ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                ctypes.POINTER(_Cache), ctypes.POINTER(_List), ctypes.c_int32,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_int32, ctypes.c_double, ctypes.c_void_p, ctypes.c_int32,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int32]
            lib.oracle_mxfp8_epilogue.restype = ctypes.c_int
            lib.oracle_mxfp8_epilogue.argtypes = [
                ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
            _lib = lib
    return _lib


def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(code & 0xFF)


def e2m1_value(nibble: int) -> float:
    return _load().oracle_e2m1_value(nibble & 0xF)


def ue8m0_value(byte: int) -> float:
    return _load().oracle_ue8m0_value(byte & 0xFF)


def e4m3_encode(y: float) -> int:
    """Nearest e4m3 code (ties to even, saturating at 448, sign kept)."""
    return int(_load().oracle_e4m3_encode(float(y)))


def ue8m0_ceil(v: float) -> int:
    """ue8m0 byte of the smallest power of two >= the fp32 value v."""
    return int(_load().oracle_ue8m0_ceil(float(v)))


def dequant_record(record: np.ndarray, fmt: int) -> np.ndarray:
    rec = np.ascontiguousarray(record, dtype=np.uint8)
    assert rec.size == RECORD_BYTES[fmt]
    out = np.zeros(KEY_DIMS.get(fmt, 512), dtype=np.float64)
    _load().oracle_dequant_record(rec.ctypes.data, fmt, out.ctypes.data)
    return out


def _np(x, dtype):
    """torch CPU tensor or numpy array -> contiguous numpy array of `dtype`
    (same-width integer types are reinterpreted, e.g. bf16 bits -> uint16)."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        x = x.detach().cpu()
        if x.dtype == torch.bfloat16:
            x = x.view(torch.int16)
        x = x.contiguous().numpy()
    a = np.ascontiguousarray(x)
    want = np.dtype(dtype)
    if a.dtype == want:
        return a
    if a.dtype.itemsize == want.itemsize and a.dtype.kind in "iu" and want.kind in "iu":
        return a.view(want)
    return a.astype(want)


def decode(q, caches, lists, *, scale: float, sink=None, positions=None, cos_sin=None,
           tokens=None, nthreads: int | None = None, rope_style: int = ROPE_NEOX):
    """Run the oracle.

    q        : bf16 [T, H, 512] (torch CPU tensor) or uint16 numpy bit patterns;
               [T, H, 576] when the lists hold V3.2 records (no RoPE then).
    caches   : sequence of dicts {bytes: uint8 array (whole cache), num_pages,
               page_size, page_stride, format} -- one per list.
    lists    : sequence of dicts {ids: int32 [T, >=width], lens: int32 [T], width}.
    sink     : fp32 [H] or None. positions: int64 [T]; cos_sin: fp32 [P, 64] or None.
    tokens   : token indices to evaluate (default: all).
    rope_style: ROPE_NEOX (dim 448+i pairs with 480+i) or ROPE_GPTJ (448+2i
               with 449+2i).
    Returns (out fp64 [n, H, 512], lse fp64 [n, H], kept int32 [n], checksum uint32 [n]).
    """
    lib = _load()
    qn = _np(q, np.uint16)
    T, H, D = qn.shape
    assert D == (576 if any(int(c["format"]) == FMT_V32_656 for c in caches) else 512)
    if tokens is None:
        tokens = np.arange(T, dtype=np.int32)
    tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    n = tok.size
    keep = []  # holds numpy arrays alive for the call
    nl = len(lists)
    assert nl == len(caches) and nl in (1, 2)
    c_arr = (_Cache * nl)()
    l_arr = (_List * nl)()
    for i, (c, l) in enumerate(zip(caches, lists)):
        b = _np(c["bytes"], np.uint8)
        keep.append(b)
        c_arr[i].base = b.ctypes.data
        c_arr[i].num_pages = int(c["num_pages"])
        c_arr[i].page_stride = int(c["page_stride"])
        c_arr[i].page_size = int(c["page_size"])
        c_arr[i].format = int(c["format"])
        need = (int(c["num_pages"]) - 1) * int(c["page_stride"]) + \
            int(c["page_size"]) * RECORD_BYTES[int(c["format"])]
        assert b.size >= need, "cache bytes shorter than its declared geometry"
        ids = _np(l["ids"], np.int32)
        lens = _np(l["lens"], np.int32)
        keep += [ids, lens]
        assert ids.shape[0] == T and lens.shape[0] == T and ids.shape[1] >= int(l["width"])
        l_arr[i].ids = ids.ctypes.data
        l_arr[i].lens = lens.ctypes.data
        l_arr[i].row_stride = ids.shape[1]
        l_arr[i].width = int(l["width"])
    sk = _np(sink, np.float32)
    pos = _np(positions, np.int64)
    cs = _np(cos_sin, np.float32)
    if cs is not None:
        assert cs.ndim == 2 and cs.shape[1] == 64
    keep += [sk, pos, cs]
    out = np.zeros((n, H, 512), dtype=np.float64)
    lse = np.zeros((n, H), dtype=np.float64)
    kept = np.zeros(n, dtype=np.int32)
    chk = np.zeros(n, dtype=np.uint32)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = lib.oracle_decode(
        H, qn.ctypes.data, qn.strides[0] // 2, qn.strides[1] // 2, c_arr, l_arr, nl,
        sk.ctypes.data if sk is not None else None,
        pos.ctypes.data if pos is not None else None,
        cs.ctypes.data if cs is not None else None,
        cs.shape[0] if cs is not None else 0, int(rope_style),
        float(scale), tok.ctypes.data, n,
        out.ctypes.data, lse.ctypes.data, kept.ctypes.data, chk.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_decode rejected its arguments")
    return out, lse, kept, chk


def mxfp8_epilogue(out, *, group_size: int, positions=None, cos_sin=None,
                   rope_style: int = ROPE_GPTJ):
    """V4.1 output epilogue of fp64 outputs out [n, H, 512] (rows of decode's
    out): inverse RoPE of dims >= 448 (when cos_sin is given; positions [n]
    are the rows' positions), fp32 rounding, MXFP8 cast (one ue8m0 scale per
    head and 32 dims), o-fused layout with `group_size` heads per group.
    Returns (codes uint8 [n, H/G, G*512], scales uint8 [n, H/G, G*16],
    x fp32 [n, H, 512] -- the values the cast was applied to)."""
    o = np.ascontiguousarray(out, dtype=np.float64)
    n, H, D = o.shape
    assert D == 512 and H % group_size == 0
    G = int(group_size)
    pos = _np(positions, np.int64)
    cs = _np(cos_sin, np.float32)
    if cs is not None:
        assert cs.ndim == 2 and cs.shape[1] == 64 and pos is not None and pos.shape == (n,)
    codes = np.zeros((n, H // G, G * 512), dtype=np.uint8)
    scales = np.zeros((n, H // G, G * 16), dtype=np.uint8)
    x = np.zeros((n, H, 512), dtype=np.float32)
    rc = _load().oracle_mxfp8_epilogue(
        o.ctypes.data, n, H, pos.ctypes.data if pos is not None else None,
        cs.ctypes.data if cs is not None else None, cs.shape[0] if cs is not None else 0,
        int(rope_style), G, x.ctypes.data, codes.ctypes.data, scales.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_mxfp8_epilogue rejected its arguments")
    return codes, scales, x


def combine(parts_out, parts_lse, sink=None):
    """Merge split-KV partials of one set of (token, head) rows.

    parts_out: [S, ..., 512] normalised partial outputs (each computed without
    a sink); parts_lse: [S, ...] their natural-log LSEs (-inf = empty part).
    Returns (out, lse): lse = log sum_i e^{lse_i};
    out = sum_i e^{lse_i} O_i / (sum_i e^{lse_i} + e^{sink}).
    """
    o = np.asarray(parts_out, dtype=np.float64)
    l = np.asarray(parts_lse, dtype=np.float64)
    m = np.max(l, axis=0)
    finite = np.isfinite(m)
    msafe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(l), np.exp(l - msafe), 0.0)
    z = w.sum(axis=0)
    lse = np.where(finite, msafe + np.log(np.where(z > 0, z, 1.0)), -np.inf)
    if sink is None:
        den = z
    else:
        sk = np.broadcast_to(np.asarray(sink, dtype=np.float64), z.shape)
        den = z + np.exp(np.minimum(sk - msafe, 700.0))
        den = np.where(np.isposinf(sk), np.inf, den)
    num = (w[..., None] * o).sum(axis=0)
    with np.errstate(invalid="ignore", divide="ignore"):
        out = np.where((den > 0)[..., None] & np.isfinite(den)[..., None],
                       num / np.where(den > 0, den, 1.0)[..., None], 0.0)
    return out, lse
