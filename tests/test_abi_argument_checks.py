"""The C ABI's argument checks, on the CPU.

Every entry point in include/w12.h validates its arguments (descriptor,
sizes, enums, null and misaligned pointers, workspace size) before it
touches the CUDA runtime, and documents the status it returns.  These
cases call libw12.so directly with a real host-encoded descriptor and fake
device addresses: each returns before any device access, so they run
without a GPU.  (Calls whose arguments are valid reach the runtime and are
covered by the -m gpu tests.)
"""
import ctypes

import numpy as np
import pytest

from lossless_bit_weight_w12_gb300 import synth

DEV = 0x7F0000000000  # a 256-byte aligned stand-in for a device address; never dereferenced


@pytest.fixture(scope="module")
def w12():
    from lossless_bit_weight_w12_gb300 import build_lib, w12 as mod
    build_lib.build()
    mod.lib()
    return mod


@pytest.fixture(scope="module")
def desc(w12):
    w = synth.weights(synth.streams(5, 1)[0], 256, 130)  # [N, K]: two column tiles, one ragged
    d, _ = w12.encode(w, w12.LAYOUT_NK)
    return d


def _c(d):
    return ctypes.byref(d.c())


def _empty_desc(w12, K, N):
    d, _ = w12.encode(np.zeros((N, K), dtype=np.uint16), w12.LAYOUT_NK)
    return d


def test_gemm_checks(w12, desc):
    L = w12.lib()
    F32, BF16 = w12.F32, w12.BF16

    def gemm(d=desc, blob=DEV, x=DEV, M=4, y=DEV, dt=F32, ws=DEV, wsb=1 << 20, path=0):
        return L.w12_gemm_ex(_c(d), blob, x, M, y, dt, ws, wsb, path, None)

    assert gemm(M=0) == w12.ERR_SHAPE
    assert gemm(M=w12.MAX_M + 1) == w12.ERR_SHAPE
    assert gemm(dt=7) == w12.ERR_ARG
    assert gemm(path=9) == w12.ERR_ARG
    assert gemm(path=-1) == w12.ERR_ARG
    assert gemm(path=0x200) == w12.ERR_ARG  # an unknown option bit
    assert gemm(path=w12.OPT_EARLY_WEIGHTS | 9) == w12.ERR_ARG
    assert gemm(y=None) == w12.ERR_ARG
    assert gemm(y=DEV + 2, dt=F32) == w12.ERR_ALIGN  # fp32 y: 4-byte aligned
    assert gemm(y=DEV + 1, dt=BF16) == w12.ERR_ALIGN  # bf16 y: 2-byte aligned
    assert gemm(blob=None) == w12.ERR_ARG
    assert gemm(x=None) == w12.ERR_ARG
    assert gemm(blob=DEV + 128) == w12.ERR_ALIGN  # blob: 256-byte aligned
    assert gemm(x=DEV + 8) == w12.ERR_ALIGN  # x: 16-byte aligned
    # a matrix with no columns: nothing to do, no pointer is looked at
    assert L.w12_gemm_ex(_c(_empty_desc(w12, 256, 0)), None, None, 4, None, F32, None, 0, 0, None) == w12.OK


def test_gemm_rejects_a_bad_descriptor(w12, desc):
    L = w12.lib()
    c = desc.c()
    c.version = 1  # an earlier format
    assert L.w12_gemm_ex(ctypes.byref(c), DEV, DEV, 4, DEV, w12.F32, DEV, 1 << 20, 0, None) != w12.OK
    c = desc.c()
    c.total_bytes += 16  # inconsistent with K, N and the escape count
    assert L.w12_gemm_ex(ctypes.byref(c), DEV, DEV, 4, DEV, w12.F32, DEV, 1 << 20, 0, None) != w12.OK


def test_batched_gemm_checks(w12, desc):
    L = w12.lib()
    arr = (type(desc.c()) * 1)(desc.c())
    ptrs = (ctypes.c_void_p * 1)(DEV)
    assert L.w12_gemm_batched_ex(arr, None, ptrs, 4, ptrs, w12.F32, 1, DEV, 1 << 20, 0, None) == w12.ERR_ARG
    assert L.w12_gemm_batched_ex(arr, ptrs, ptrs, 4, ptrs, 5, 1, DEV, 1 << 20, 0, None) == w12.ERR_ARG
    assert L.w12_gemm_batched_ex(arr, ptrs, ptrs, 4, ptrs, w12.F32, 1, DEV, 1 << 20, 7, None) == w12.ERR_ARG
    assert L.w12_gemm_batched_ex(arr, ptrs, ptrs, 4, ptrs, w12.F32, 1, DEV, 1 << 20, 0x400, None) == w12.ERR_ARG


def test_batched_debug_checks(w12, desc):
    """The test-hook entry point rejects a missing or out-of-range hook
    before it looks at anything else."""
    L = w12.lib()
    arr = (type(desc.c()) * 1)(desc.c())
    ptrs = (ctypes.c_void_p * 1)(DEV)

    def dbg_call(dbg, path=0):
        return L.w12_gemm_batched_debug(arr, ptrs, ptrs, 4, ptrs, w12.F32, 1, DEV, 1 << 20, path,
                                        dbg, None)
    assert dbg_call(None) == w12.ERR_ARG
    assert dbg_call(ctypes.byref(w12._CDebug(-2, 0))) == w12.ERR_ARG
    assert dbg_call(ctypes.byref(w12._CDebug(-1, 20_000_000))) == w12.ERR_ARG
    assert dbg_call(ctypes.byref(w12._CDebug(-1, 0)), path=9) == w12.ERR_ARG


def test_decode_checks(w12, desc):
    L = w12.lib()
    assert L.w12_decode(_c(desc), DEV, DEV, 5, None, None) == w12.ERR_ARG
    assert L.w12_decode(_c(desc), None, DEV, w12.LAYOUT_NK, None, None) == w12.ERR_ARG
    assert L.w12_decode(_c(desc), DEV, None, w12.LAYOUT_NK, None, None) == w12.ERR_ARG
    assert L.w12_decode(_c(desc), DEV + 16, DEV, w12.LAYOUT_NK, None, None) == w12.ERR_ALIGN
    assert L.w12_decode(_c(desc), DEV, DEV + 4, w12.LAYOUT_NK, None, None) == w12.ERR_ALIGN
    assert L.w12_decode(_c(_empty_desc(w12, 0, 64)), None, None, w12.LAYOUT_NK, None, None) == w12.OK


@pytest.mark.parametrize("noalloc", [False, True])
def test_verify_checks(w12, noalloc):
    L = w12.lib()

    def verify(lg=DEV, dt=0, R=1, T=16, V=4096, draft=DEV, acc=DEV, nxt=DEV):
        if noalloc:
            return L.w12_verify_greedy_noalloc(lg, dt, R, T, V, draft, acc, nxt, None)
        return L.w12_verify_greedy(lg, dt, R, T, V, draft, acc, nxt, DEV, 1 << 20, None)

    assert verify(dt=3) == w12.ERR_ARG
    assert verify(R=0) == w12.ERR_SHAPE
    assert verify(T=0) == w12.ERR_SHAPE
    assert verify(V=0) == w12.ERR_SHAPE
    assert verify(V=1 << 31) == w12.ERR_SHAPE
    assert verify(lg=None) == w12.ERR_ARG
    assert verify(draft=None) == w12.ERR_ARG  # T > 1 needs drafts
    assert verify(acc=None) == w12.ERR_ARG
    assert verify(nxt=None) == w12.ERR_ARG
    assert verify(lg=DEV + 2, dt=w12.F32) == w12.ERR_ALIGN
    assert verify(lg=DEV + 1, dt=w12.BF16) == w12.ERR_ALIGN
    assert verify(acc=DEV + 2) == w12.ERR_ALIGN
    assert verify(draft=DEV + 2) == w12.ERR_ALIGN
    assert L.w12_verify_workspace_size(0, 16, 4096) == 0
    assert L.w12_verify_workspace_size(1, 16, 1 << 31) == 0


def test_verify_lmhead_checks(w12, desc):
    L = w12.lib()

    def vl(h=DEV, d=desc, blob=DEV, R=1, T=16, draft=DEV, acc=DEV, nxt=DEV, lo=None):
        return L.w12_verify_greedy_lmhead(h, _c(d), blob, R, T, draft, acc, nxt, lo, DEV, 1 << 24, None)

    assert vl(R=0) == w12.ERR_SHAPE
    assert vl(R=9, T=16) == w12.ERR_SHAPE  # R * T > W12_MAX_M
    assert vl(h=None) == w12.ERR_ARG
    assert vl(blob=None) == w12.ERR_ARG
    assert vl(draft=None) == w12.ERR_ARG
    assert vl(blob=DEV + 64) == w12.ERR_ALIGN
    assert vl(h=DEV + 8) == w12.ERR_ALIGN
    assert vl(lo=DEV + 2) == w12.ERR_ALIGN
    assert L.w12_verify_lmhead_workspace_size(_c(desc), 9, 16) == 0


def test_device_encoder_checks(w12, desc):
    L = w12.lib()
    c = type(desc.c())()
    ws = L.w12_encode_device_workspace_size(256, 130)
    assert ws > 0
    assert L.w12_encode_plan_device(DEV, 256, 130, 7, ctypes.byref(c), DEV, ws, None) == w12.ERR_ARG
    assert L.w12_encode_plan_device(DEV, 200, 130, w12.LAYOUT_NK, ctypes.byref(c), DEV, ws, None) == w12.ERR_SHAPE
    assert L.w12_encode_plan_device(None, 256, 130, w12.LAYOUT_NK, ctypes.byref(c), DEV, ws, None) == w12.ERR_ARG
    assert L.w12_encode_plan_device(DEV + 8, 256, 130, w12.LAYOUT_NK, ctypes.byref(c), DEV, ws,
                                    None) == w12.ERR_ALIGN
    assert L.w12_encode_plan_device(DEV, 256, 130, w12.LAYOUT_NK, ctypes.byref(c), DEV, ws - 1,
                                    None) == w12.ERR_WORKSPACE
    # an empty matrix is planned without touching the device
    assert L.w12_encode_plan_device(None, 0, 130, w12.LAYOUT_NK, ctypes.byref(c), None, 0, None) == w12.OK
    assert c.total_bytes == 0
    # encode: the descriptor must be the one planned for these K, N
    assert L.w12_encode_device(DEV, 256, 131, w12.LAYOUT_NK, _c(desc), DEV, DEV, ws, None) == w12.ERR_ARG
    assert L.w12_encode_device(DEV, 256, 130, 9, _c(desc), DEV, DEV, ws, None) == w12.ERR_ARG
    assert L.w12_encode_device(DEV, 256, 130, w12.LAYOUT_NK, _c(desc), DEV + 16, DEV, ws, None) == w12.ERR_ALIGN
    assert L.w12_encode_device(DEV, 256, 130, w12.LAYOUT_NK, _c(desc), DEV, DEV, ws - 1,
                               None) == w12.ERR_WORKSPACE
