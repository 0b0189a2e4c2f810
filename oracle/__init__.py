"""CPU oracle for the INT4 + 2:4 "2bit-CSR" SparseGemv -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import this
package. The product (``int4_weight_only_sgemv_gb300``) never imports it and shares no code with it.

The oracle itself is plain C++17 in ``oracle.cpp`` (pack, dequantise and an fp64 GEMV written from the
packed-format definition, one element at a time). This module compiles it with g++ and wraps it with
ctypes and numpy. Method source: the paper "Efficient LLM-based Advertising via Model Compression and
Parallel Verification", §3.2 (group-wise INT4 quantisation, 2:4 pruning) and §3.3 (2bit-CSR index,
SparseGemv).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

FMT_SPARSE24 = 1
FMT_DENSE = 2
FMT_SPARSE14 = 3


def build(force: bool = False) -> str:
    """Compile oracle.cpp into oracle/_build/liboracle.so (OpenMP if the compiler has it)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    base = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared", _SRC]
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    try:
        subprocess.run(base + ["-fopenmp", "-o", tmp], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-o", tmp], check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            u8p = ctypes.POINTER(ctypes.c_uint8)
            u16p = ctypes.POINTER(ctypes.c_uint16)
            u64p = ctypes.POINTER(ctypes.c_uint64)
            i32p = ctypes.POINTER(ctypes.c_int32)
            f64p = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            L.orc_half_to_float.argtypes = [ctypes.c_uint16]
            L.orc_half_to_float.restype = ctypes.c_float
            L.orc_float_to_half.argtypes = [ctypes.c_float]
            L.orc_float_to_half.restype = ctypes.c_uint16
            L.orc_layout.argtypes = [ctypes.c_int, i64, i64, i64, u64p]
            L.orc_pack.argtypes = [ctypes.c_int, i64, i64, i64, u16p, u8p, ctypes.c_uint64]
            L.orc_dequant.argtypes = [u8p, ctypes.c_uint64, f64p]
            L.orc_unpack.argtypes = [u8p, ctypes.c_uint64, u8p, i32p, u16p, u16p]
            L.orc_gemv_rows.argtypes = [u8p, ctypes.c_uint64, u16p, ctypes.c_int, i32p, i64, f64p,
                                        f64p, ctypes.c_int]
            L.orc_gemv.argtypes = [u8p, ctypes.c_uint64, u16p, ctypes.c_int, f64p, f64p, ctypes.c_int]
            L.orc_openmp_available.argtypes = []
            for name in ("orc_layout", "orc_pack", "orc_dequant", "orc_unpack", "orc_gemv_rows",
                         "orc_gemv", "orc_openmp_available"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what} failed with status {code}")
        self.code = code


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _h16(a) -> np.ndarray:
    """fp16 data as a contiguous uint16 view."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("expected float16 or uint16 bits")
    return a


def half_to_float(h: int) -> float:
    return lib().orc_half_to_float(int(h))


def float_to_half(f: float) -> int:
    return lib().orc_float_to_half(float(f))


def layout(fmt: int, n: int, k: int, g: int) -> dict:
    out = np.zeros(9, dtype=np.uint64)
    rc = lib().orc_layout(fmt, n, k, g, _ptr(out, ctypes.c_uint64))
    if rc != 0:
        raise OracleError(rc, "orc_layout")
    keys = ("vals_pitch", "idx_pitch", "sz_pitch", "off_vals", "off_idx", "off_sz", "off_rowptr",
            "total_bytes", "kept_per_row")
    return {k_: int(v) for k_, v in zip(keys, out)}


def pack(w, fmt: int, g: int) -> np.ndarray:
    """Pack fp16 W[n][k]; returns the packed bytes (uint8, length total_bytes)."""
    w = _h16(w)
    n, k = w.shape
    L = layout(fmt, n, k, g)
    out = np.empty(L["total_bytes"], dtype=np.uint8)
    rc = lib().orc_pack(fmt, n, k, g, _ptr(w, ctypes.c_uint16), _ptr(out, ctypes.c_uint8), out.size)
    if rc != 0:
        raise OracleError(rc, "orc_pack")
    return out


def header(buf: np.ndarray) -> dict:
    b = np.ascontiguousarray(buf, dtype=np.uint8)
    u32 = b[:24].view(np.uint32)
    u64 = b[24:64].view(np.uint64)
    return {"magic": int(u32[0]), "version": int(u32[1]), "format": int(u32[2]), "n": int(u32[3]),
            "k": int(u32[4]), "g": int(u32[5]), "off_vals": int(u64[0]), "off_idx": int(u64[1]),
            "off_sz": int(u64[2]), "off_rowptr": int(u64[3]), "total_bytes": int(u64[4])}


def dequant(buf: np.ndarray) -> np.ndarray:
    """Dense fp64 Ŵ[n][k] decoded from a packed buffer."""
    h = header(buf)
    out = np.empty((h["n"], h["k"]), dtype=np.float64)
    rc = lib().orc_dequant(_ptr(buf, ctypes.c_uint8), buf.size, _ptr(out, ctypes.c_double))
    if rc != 0:
        raise OracleError(rc, "orc_dequant")
    return out


def unpack(buf: np.ndarray) -> dict:
    """Per-row kept nibbles q, dense columns col, and per-group s16/z16 bits."""
    h = header(buf)
    n, k, g = h["n"], h["k"], h["g"]
    kpr = {FMT_SPARSE24: k // 2, FMT_SPARSE14: k // 4}.get(h["format"], k)
    q = np.empty((n, kpr), dtype=np.uint8)
    col = np.empty((n, kpr), dtype=np.int32)
    s16 = np.empty((n, k // g), dtype=np.uint16)
    z16 = np.empty((n, k // g), dtype=np.uint16)
    rc = lib().orc_unpack(_ptr(buf, ctypes.c_uint8), buf.size, _ptr(q, ctypes.c_uint8),
                          _ptr(col, ctypes.c_int32), _ptr(s16, ctypes.c_uint16), _ptr(z16, ctypes.c_uint16))
    if rc != 0:
        raise OracleError(rc, "orc_unpack")
    return {"q": q, "col": col, "s16": s16, "z16": z16}


def gemv(buf: np.ndarray, x, rows=None, nthreads: int = 1):
    """fp64 y[b][r] and Σ|ŵ·x|[b][r] for all rows, or for the listed rows only."""
    x = _h16(x)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    batch = x.shape[0]
    if rows is None:
        nr = header(buf)["n"]
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int32)
        nr = rows_arr.size
    y = np.empty((batch, nr), dtype=np.float64)
    absdot = np.empty((batch, nr), dtype=np.float64)
    rc = lib().orc_gemv_rows(_ptr(buf, ctypes.c_uint8), buf.size, _ptr(x, ctypes.c_uint16), batch,
                             None if rows_arr is None else _ptr(rows_arr, ctypes.c_int32), nr,
                             _ptr(y, ctypes.c_double), _ptr(absdot, ctypes.c_double), int(nthreads))
    if rc != 0:
        raise OracleError(rc, "orc_gemv_rows")
    return y, absdot


def openmp_available() -> bool:
    return bool(lib().orc_openmp_available())
