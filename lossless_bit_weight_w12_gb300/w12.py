"""Thin ctypes binding of libw12.so (include/w12.h), same names as the C calls.

Argument marshalling only: host arrays are numpy, device buffers are torch
CUDA tensors (used for their memory and streams); every computation runs in
the library's kernels or its host encoder.  The library is loaded on first
use from ``lossless_bit_weight_w12_gb300/_build/libw12.so``; if it is missing
this raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libw12.so")

OK = 0
ERR_ARG, ERR_SHAPE, ERR_ALIGN, ERR_WORKSPACE, ERR_BLOB = 1, 2, 3, 4, 5
ERR_TOO_MANY_ESCAPES, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE = 6, 7, 8, 9
LAYOUT_KN, LAYOUT_NK = 0, 1
F32, BF16 = 0, 1
PATH_AUTO, PATH_GEMV, PATH_MMA, PATH_TC = 0, 1, 2, 3
OPT_EARLY_WEIGHTS = 0x100  # OR into a path: weight copies start under the previous kernel's tail
MAX_M = 128

# every symbol include/w12.h declares
EXPORTS = (
    "w12_status_string", "w12_version", "w12_encode_plan", "w12_encode", "w12_validate",
    "w12_decode", "w12_gemm_workspace_size", "w12_gemm", "w12_gemm_ex",
    "w12_verify_workspace_size", "w12_verify_greedy", "w12_verify_lmhead_workspace_size",
    "w12_verify_greedy_lmhead", "w12_get_device_error", "w12_verify_greedy_noalloc",
    "w12_gemm_batched_workspace_size", "w12_gemm_batched", "w12_gemm_batched_ex",
    "w12_encode_device_workspace_size", "w12_encode_plan_device", "w12_encode_device",
    "w12_gemm_batched_debug",
)


class W12Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)}")
        self.status = status


class _CDesc(ctypes.Structure):
    _fields_ = [("version", ctypes.c_uint32), ("reserved", ctypes.c_uint32),
                ("K", ctypes.c_int64), ("N", ctypes.c_int64), ("G", ctypes.c_int64),
                ("tiles", ctypes.c_uint64), ("unit_bytes", ctypes.c_uint64),
                ("n_units", ctypes.c_uint64), ("off_units", ctypes.c_uint64),
                ("off_esc", ctypes.c_uint64), ("n_esc", ctypes.c_uint64),
                ("total_bytes", ctypes.c_uint64)]


class _CDebug(ctypes.Structure):
    _fields_ = [("withhold_unit", ctypes.c_int32), ("wait_limit_us", ctypes.c_uint32)]


@dataclass(frozen=True)
class Desc:
    """w12_desc of one encoded K x N matrix."""
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

    def c(self) -> _CDesc:
        return _CDesc(self.version, 0, self.K, self.N, self.G, self.tiles, self.unit_bytes,
                      self.n_units, self.off_units, self.off_esc, self.n_esc, self.total_bytes)

    @staticmethod
    def from_c(c: _CDesc) -> "Desc":
        return Desc(c.version, c.K, c.N, c.G, c.tiles, c.unit_bytes, c.n_units, c.off_units,
                    c.off_esc, c.n_esc, c.total_bytes)


_lib = None


def lib():
    """Load libw12.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libw12.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        D = ctypes.POINTER(_CDesc)
        L.w12_status_string.restype = ctypes.c_char_p
        L.w12_status_string.argtypes = [I]
        L.w12_version.argtypes = []
        L.w12_encode_plan.argtypes = [P, I64, I64, I, D]
        L.w12_encode.argtypes = [P, I64, I64, I, D, P]
        L.w12_validate.argtypes = [D, P]
        L.w12_decode.argtypes = [D, P, P, I, P, P]
        L.w12_gemm_workspace_size.restype = SZ
        L.w12_gemm_workspace_size.argtypes = [D, I64]
        L.w12_gemm.argtypes = [D, P, P, I64, P, I, P, SZ, P]
        L.w12_gemm_ex.argtypes = [D, P, P, I64, P, I, P, SZ, I, P]
        L.w12_verify_workspace_size.restype = SZ
        L.w12_verify_workspace_size.argtypes = [I64, I64, I64]
        L.w12_verify_greedy.argtypes = [P, I, I64, I64, I64, P, P, P, P, SZ, P]
        L.w12_verify_lmhead_workspace_size.restype = SZ
        L.w12_verify_lmhead_workspace_size.argtypes = [D, I64, I64]
        L.w12_verify_greedy_lmhead.argtypes = [P, D, P, I64, I64, P, P, P, P, P, SZ, P]
        L.w12_get_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_int), P]
        L.w12_verify_greedy_noalloc.argtypes = [P, I, I64, I64, I64, P, P, P, P]
        L.w12_gemm_batched_workspace_size.restype = SZ
        L.w12_gemm_batched_workspace_size.argtypes = [D, I, I64]
        L.w12_gemm_batched.argtypes = [D, P, P, I64, P, I, I, P, SZ, P]
        L.w12_gemm_batched_ex.argtypes = [D, P, P, I64, P, I, I, P, SZ, I, P]
        L.w12_encode_device_workspace_size.restype = SZ
        L.w12_encode_device_workspace_size.argtypes = [I64, I64]
        L.w12_encode_plan_device.argtypes = [P, I64, I64, I, D, P, SZ, P]
        L.w12_encode_device.argtypes = [P, I64, I64, I, D, P, P, SZ, P]
        L.w12_gemm_batched_debug.argtypes = [D, P, P, I64, P, I, I, P, SZ, I, ctypes.POINTER(_CDebug), P]
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().w12_status_string(status).decode()


def version() -> int:
    return lib().w12_version()


def _check(st: int, what: str):
    if st != OK:
        raise W12Error(st, what)


def _np_ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _dptr(t):
    """Device pointer of a torch CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _kn(w, layout):
    return (w.shape[0], w.shape[1]) if layout == LAYOUT_KN else (w.shape[1], w.shape[0])


# --------------------------------------------------------------------- host

def encode_plan(w: np.ndarray, layout: int = LAYOUT_NK) -> Desc:
    w = np.ascontiguousarray(w, dtype=np.uint16)
    K, N = _kn(w, layout)
    c = _CDesc()
    _check(lib().w12_encode_plan(_np_ptr(w), K, N, layout, ctypes.byref(c)), "w12_encode_plan")
    return Desc.from_c(c)


def encode(w: np.ndarray, layout: int = LAYOUT_NK, desc: Desc | None = None):
    """Encode bf16 bit patterns w on the host; returns (Desc, blob uint8 array)."""
    w = np.ascontiguousarray(w, dtype=np.uint16)
    K, N = _kn(w, layout)
    d = desc if desc is not None else encode_plan(w, layout)
    blob = np.empty(d.total_bytes, dtype=np.uint8)
    c = d.c()
    _check(lib().w12_encode(_np_ptr(w), K, N, layout, ctypes.byref(c), _np_ptr(blob)),
           "w12_encode")
    return d, blob


def validate(d: Desc, blob: np.ndarray) -> int:
    """Returns the status (OK or ERR_BLOB / ERR_ARG) without raising."""
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    c = d.c()
    return lib().w12_validate(ctypes.byref(c), _np_ptr(blob))


# ------------------------------------------------------------------- device

def decode(d: Desc, blob_dev, w_dev, layout: int = LAYOUT_NK, err_dev=None, stream=None):
    c = d.c()
    _check(lib().w12_decode(ctypes.byref(c), _dptr(blob_dev), _dptr(w_dev), layout,
                            _dptr(err_dev), _stream(stream)), "w12_decode")


def encode_device(w_dev, layout: int = LAYOUT_NK, stream=None):
    """Encode bf16 bit patterns already on the device (a torch int16/uint16
    CUDA tensor, [N, K] for LAYOUT_NK or [K, N] for LAYOUT_KN) on the GPU;
    returns (Desc, blob device tensor, 256-byte aligned)."""
    import torch
    K, N = _kn(w_dev, layout)
    ws = workspace(lib().w12_encode_device_workspace_size(K, N), w_dev.device)
    c = _CDesc()
    _check(lib().w12_encode_plan_device(_dptr(w_dev), K, N, layout, ctypes.byref(c), _dptr(ws), ws.numel(),
                                        _stream(stream)), "w12_encode_plan_device")
    d = Desc.from_c(c)
    t = torch.empty(d.total_bytes + 256, dtype=torch.uint8, device=w_dev.device)
    off = (-t.data_ptr()) % 256
    blob = t[off:off + d.total_bytes]
    if d.total_bytes:
        c = d.c()
        _check(lib().w12_encode_device(_dptr(w_dev), K, N, layout, ctypes.byref(c), _dptr(blob), _dptr(ws),
                                       ws.numel(), _stream(stream)), "w12_encode_device")
    return d, blob


def gemm_workspace_size(d: Desc, M: int) -> int:
    c = d.c()
    return int(lib().w12_gemm_workspace_size(ctypes.byref(c), M))


def gemm(d: Desc, blob_dev, x_dev, y_dev, ws_dev, path: int = PATH_AUTO, stream=None):
    """y_dev[M, N] (float32 or bfloat16) = x_dev[M, K] (bfloat16) @ W."""
    import torch
    M = x_dev.shape[0]
    y_dtype = F32 if y_dev.dtype == torch.float32 else BF16
    c = d.c()
    _check(lib().w12_gemm_ex(ctypes.byref(c), _dptr(blob_dev), _dptr(x_dev), M, _dptr(y_dev),
                             y_dtype, _dptr(ws_dev), ws_dev.numel() * ws_dev.element_size(),
                             path, _stream(stream)), "w12_gemm")


def _desc_array(descs):
    arr = (_CDesc * len(descs))()
    for i, d in enumerate(descs):
        arr[i] = d.c()
    return arr


def gemm_batched_workspace_size(descs, M: int) -> int:
    return int(lib().w12_gemm_batched_workspace_size(_desc_array(descs), len(descs), M))


class GemmBatch:
    """Marshalled arguments of one w12_gemm_batched call (built once, reused:
    the pointer arrays stay valid while the tensors live)."""

    def __init__(self, descs, blobs, xs, ys, ws, path: int = PATH_AUTO):
        import torch
        n = len(descs)
        self.path = path
        self.descs = _desc_array(descs)
        self.blobs = (ctypes.c_void_p * n)(*[t.data_ptr() for t in blobs])
        self.xs = (ctypes.c_void_p * n)(*[t.data_ptr() for t in xs])
        self.ys = (ctypes.c_void_p * n)(*[t.data_ptr() for t in ys])
        self.M = xs[0].shape[0]
        self.y_dtype = F32 if ys[0].dtype == torch.float32 else BF16
        self.count = n
        self.ws = ws
        self._keep = (blobs, xs, ys, ws)

    def __call__(self, stream=None):
        _check(lib().w12_gemm_batched_ex(self.descs, self.blobs, self.xs, self.M, self.ys,
                                         self.y_dtype, self.count, _dptr(self.ws),
                                         self.ws.numel() * self.ws.element_size(), self.path,
                                         _stream(stream)),
               "w12_gemm_batched_ex")


def gemm_batched(descs, blobs, xs, ys, ws, path: int = PATH_AUTO, stream=None):
    """ys[i] = xs[i] @ W_i for every i, in one launch."""
    GemmBatch(descs, blobs, xs, ys, ws, path)(stream)


def gemm_batched_debug(descs, blobs, xs, ys, ws, withhold_unit: int = -1, wait_limit_us: int = 0,
                       path: int = PATH_AUTO, stream=None):
    """w12_gemm_batched_debug: the batched GEMM with the test hooks (a
    withheld weight copy, a short wait limit)."""
    b = GemmBatch(descs, blobs, xs, ys, ws, path)
    dbg = _CDebug(withhold_unit, wait_limit_us)
    _check(lib().w12_gemm_batched_debug(b.descs, b.blobs, b.xs, b.M, b.ys, b.y_dtype, b.count, _dptr(ws),
                                        ws.numel() * ws.element_size(), path, ctypes.byref(dbg),
                                        _stream(stream)),
           "w12_gemm_batched_debug")


def verify_workspace_size(R: int, T: int, V: int) -> int:
    return int(lib().w12_verify_workspace_size(R, T, V))


def verify_greedy(logits_dev, R: int, T: int, draft_dev, accept_dev, next_dev, ws_dev,
                  stream=None):
    import torch
    dtype = F32 if logits_dev.dtype == torch.float32 else BF16
    V = logits_dev.shape[-1]
    _check(lib().w12_verify_greedy(_dptr(logits_dev), dtype, R, T, V, _dptr(draft_dev),
                                   _dptr(accept_dev), _dptr(next_dev), _dptr(ws_dev),
                                   ws_dev.numel() * ws_dev.element_size(), _stream(stream)),
           "w12_verify_greedy")


def verify_lmhead_workspace_size(d: Desc, R: int, T: int) -> int:
    c = d.c()
    return int(lib().w12_verify_lmhead_workspace_size(ctypes.byref(c), R, T))


def verify_greedy_lmhead(hidden_dev, d: Desc, blob_dev, R: int, T: int, draft_dev, accept_dev,
                         next_dev, ws_dev, logits_out_dev=None, stream=None):
    c = d.c()
    _check(lib().w12_verify_greedy_lmhead(_dptr(hidden_dev), ctypes.byref(c), _dptr(blob_dev),
                                          R, T, _dptr(draft_dev), _dptr(accept_dev),
                                          _dptr(next_dev), _dptr(logits_out_dev), _dptr(ws_dev),
                                          ws_dev.numel() * ws_dev.element_size(),
                                          _stream(stream)), "w12_verify_greedy_lmhead")


def verify_greedy_noalloc(logits_dev, R: int, T: int, draft_dev, accept_dev, next_dev,
                          stream=None):
    """verify_greedy() on the library's own fixed scratch array: for callers
    that cannot allocate device memory (see include/w12.h)."""
    import torch
    dtype = F32 if logits_dev.dtype == torch.float32 else BF16
    V = logits_dev.shape[-1]
    _check(lib().w12_verify_greedy_noalloc(_dptr(logits_dev), dtype, R, T, V, _dptr(draft_dev),
                                           _dptr(accept_dev), _dptr(next_dev), _stream(stream)),
           "w12_verify_greedy_noalloc")


def get_device_error(ws_dev, stream=None) -> int:
    v = ctypes.c_int(0)
    _check(lib().w12_get_device_error(_dptr(ws_dev), ctypes.byref(v), _stream(stream)),
           "w12_get_device_error")
    return v.value


# --------------------------------------------------------------- helpers

def workspace(nbytes: int, device="cuda"):
    """A zero-filled, 256-byte aligned device workspace of nbytes (torch uint8)."""
    import torch
    t = torch.zeros(max(int(nbytes), 256) + 256, dtype=torch.uint8, device=device)
    off = (-t.data_ptr()) % 256
    return t[off:off + max(int(nbytes), 256)]


def upload(blob: np.ndarray, device="cuda"):
    """Copy a host blob to a 256-byte aligned device buffer."""
    import torch
    n = blob.size
    t = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-t.data_ptr()) % 256
    t = t[off:off + n]
    t.copy_(torch.from_numpy(np.ascontiguousarray(blob)))
    return t


class Weight:
    """An encoded matrix resident on the device: desc + 256-byte aligned blob."""

    def __init__(self, w: np.ndarray, layout: int = LAYOUT_NK, device="cuda"):
        self.desc, blob = encode(w, layout)
        self.blob = upload(blob, device)

    @property
    def K(self):
        return self.desc.K

    @property
    def N(self):
        return self.desc.N
