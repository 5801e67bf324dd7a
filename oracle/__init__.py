"""CPU oracle for the W12 hot path (ctypes over oracle/w12_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product library
never does.  It shares no code with the CUDA library.

Functions (host numpy arrays in, host numpy arrays out):
  plan(w, layout)            -> Desc           (escape count, blob offsets)
  encode(w, layout)          -> (Desc, blob)   W12 v2 blob, uint8
  decode(desc, blob, layout) -> w              bf16 bit patterns, uint16
  group_base(vals128)        -> int            per-group base rule
  gemm(desc, blob, x)        -> (y, s)         fp64 y = x @ W, s = sum |x w|
  gemm_at(desc, blob, x, ms, ns) -> (y, s)     selected outputs only
  argmax(logits)             -> idx            lowest index of the row max
  verify_greedy(logits, R, T, draft) -> (accept_len, next_token)
"""
import ctypes
import os
from dataclasses import dataclass

import numpy as np

from . import build as _build

LAYOUT_KN = 0
LAYOUT_NK = 1
F32 = 0
BF16 = 1

OK = 0
ERR_ARG = 1
ERR_SHAPE = 2
ERR_BLOB = 5
ERR_TOO_MANY_ESCAPES = 6


class _CDesc(ctypes.Structure):
    _fields_ = [("version", ctypes.c_uint32), ("reserved", ctypes.c_uint32),
                ("K", ctypes.c_int64), ("N", ctypes.c_int64), ("G", ctypes.c_int64),
                ("tiles", ctypes.c_uint64), ("unit_bytes", ctypes.c_uint64),
                ("n_units", ctypes.c_uint64), ("off_units", ctypes.c_uint64),
                ("off_esc", ctypes.c_uint64), ("n_esc", ctypes.c_uint64),
                ("total_bytes", ctypes.c_uint64)]


@dataclass
class Desc:
    version: int
    K: int
    N: int
    G: int
    tiles: int
    unit_bytes: int
    n_units: int
    off_units: int
    off_esc: int
    n_esc: int
    total_bytes: int

    def _c(self) -> _CDesc:
        return _CDesc(self.version, 0, self.K, self.N, self.G, self.tiles, self.unit_bytes,
                      self.n_units, self.off_units, self.off_esc, self.n_esc, self.total_bytes)

    @staticmethod
    def _from_c(c: _CDesc) -> "Desc":
        return Desc(c.version, c.K, c.N, c.G, c.tiles, c.unit_bytes, c.n_units, c.off_units,
                    c.off_esc, c.n_esc, c.total_bytes)


class OracleError(RuntimeError):
    def __init__(self, status, what):
        super().__init__(f"oracle {what} failed with status {status}")
        self.status = status


_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        L.w12ref_group_base.argtypes = [P]
        L.w12ref_plan.argtypes = [P, I64, I64, ctypes.c_int, ctypes.POINTER(_CDesc)]
        L.w12ref_encode.argtypes = [P, I64, I64, ctypes.c_int, ctypes.POINTER(_CDesc), P]
        L.w12ref_decode.argtypes = [ctypes.POINTER(_CDesc), P, P, ctypes.c_int]
        L.w12ref_gemm.argtypes = [ctypes.POINTER(_CDesc), P, P, I64, P, P]
        L.w12ref_gemm_at.argtypes = [ctypes.POINTER(_CDesc), P, P, I64, I64, P, P, P, P]
        L.w12ref_argmax.argtypes = [P, ctypes.c_int, I64, I64, P]
        L.w12ref_verify_greedy.argtypes = [P, ctypes.c_int, I64, I64, I64, P, P, P]
        _lib = L
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _check(st, what):
    if st != OK:
        raise OracleError(st, what)


def _shape_kn(w, layout):
    if layout == LAYOUT_KN:
        return w.shape[0], w.shape[1]
    return w.shape[1], w.shape[0]


def group_base(vals) -> int:
    v = np.ascontiguousarray(vals, dtype=np.uint16)
    assert v.shape == (128,)
    return lib().w12ref_group_base(_ptr(v))


def plan(w, layout=LAYOUT_KN) -> Desc:
    w = np.ascontiguousarray(w, dtype=np.uint16)
    K, N = _shape_kn(w, layout)
    c = _CDesc()
    _check(lib().w12ref_plan(_ptr(w), K, N, layout, ctypes.byref(c)), "plan")
    return Desc._from_c(c)


def encode(w, layout=LAYOUT_KN):
    w = np.ascontiguousarray(w, dtype=np.uint16)
    K, N = _shape_kn(w, layout)
    d = plan(w, layout)
    blob = np.zeros(d.total_bytes, dtype=np.uint8)
    c = d._c()
    _check(lib().w12ref_encode(_ptr(w), K, N, layout, ctypes.byref(c), _ptr(blob)), "encode")
    return d, blob


def decode(d: Desc, blob, layout=LAYOUT_KN):
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    shape = (d.K, d.N) if layout == LAYOUT_KN else (d.N, d.K)
    w = np.zeros(shape, dtype=np.uint16)
    c = d._c()
    _check(lib().w12ref_decode(ctypes.byref(c), _ptr(blob), _ptr(w), layout), "decode")
    return w


def gemm(d: Desc, blob, x):
    """x: [M, K] bf16 bit patterns (uint16). Returns fp64 (y, s), each [M, N]."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    M = x.shape[0]
    assert x.shape[1] == d.K
    y = np.zeros((M, d.N), dtype=np.float64)
    s = np.zeros((M, d.N), dtype=np.float64)
    c = d._c()
    _check(lib().w12ref_gemm(ctypes.byref(c), _ptr(np.ascontiguousarray(blob)), _ptr(x), M,
                             _ptr(y), _ptr(s)), "gemm")
    return y, s


def gemm_at(d: Desc, blob, x, ms, ns):
    x = np.ascontiguousarray(x, dtype=np.uint16)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    assert ms.shape == ns.shape
    y = np.zeros(ms.shape, dtype=np.float64)
    s = np.zeros(ms.shape, dtype=np.float64)
    c = d._c()
    _check(lib().w12ref_gemm_at(ctypes.byref(c), _ptr(np.ascontiguousarray(blob)), _ptr(x),
                                x.shape[0], ms.size, _ptr(ms), _ptr(ns), _ptr(y), _ptr(s)),
           "gemm_at")
    return y, s


def _logits_dtype(logits):
    if logits.dtype == np.float32:
        return F32
    if logits.dtype == np.uint16:
        return BF16
    raise TypeError("logits must be float32 or bf16 bit patterns (uint16)")


def argmax(logits):
    logits = np.ascontiguousarray(logits)
    rows, V = logits.shape
    idx = np.zeros(rows, dtype=np.int64)
    _check(lib().w12ref_argmax(_ptr(logits), _logits_dtype(logits), rows, V, _ptr(idx)),
           "argmax")
    return idx


def verify_greedy(logits, R, T, draft):
    """logits: [R*T, V] float32 or bf16 bits; draft: [R, T-1] int32."""
    logits = np.ascontiguousarray(logits)
    V = logits.shape[1]
    assert logits.shape[0] == R * T
    draft = np.ascontiguousarray(draft, dtype=np.int32).reshape(R, max(T - 1, 0))
    acc = np.zeros(R, dtype=np.int32)
    nxt = np.zeros(R, dtype=np.int32)
    _check(lib().w12ref_verify_greedy(_ptr(logits), _logits_dtype(logits), R, T, V,
                                      _ptr(draft), _ptr(acc), _ptr(nxt)), "verify_greedy")
    return acc, nxt


def lib_path() -> str:
    return os.path.abspath(_build.LIB)
