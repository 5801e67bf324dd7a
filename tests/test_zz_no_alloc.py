"""w12_verify_greedy_noalloc: greedy verification for callers that cannot
allocate device memory (a serving loop whose memory is fixed at start-up, a
host framework that owns every allocation, a path that cannot afford
cudaMalloc's device synchronisation).  It runs on a scratch array the library
keeps on each GPU instead of a caller workspace.

The test calls both entry points through the C ABI (ctypes on libw12.so) on
the same device buffers and requires identical (accept_len, next_token), bit
for bit as every verify test, on two calls in a row: the second call sees the
scratch the first one left behind.  The file sorts last so a run that stops
at the first failure has already run everything else.
"""
import ctypes

import numpy as np
import pytest

from lossless_bit_weight_w12_gb300 import synth

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def test_noalloc_matches_workspace_entry_point(dev, w12mod, oracle):
    import torch
    L = w12mod.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [(1, 16, 151936, np.float32, 41), (4, 8, 32000, np.uint16, 42)]
    for R, T, V, dtype, seed in cases:  # two calls in a row, different shapes
        rng = synth.streams(seed, 2)
        lg = synth.logits(rng[0], R * T, V, dtype=dtype)
        draft = synth.draft_tokens(rng[1], oracle.argmax(lg).reshape(R, T), R, T, V)
        if dtype == np.uint16:
            lg_d = torch.from_numpy(lg.view(np.int16)).to(dev)
            code = w12mod.BF16
        else:
            lg_d = torch.from_numpy(lg).to(dev)
            code = w12mod.F32
        dr_d = torch.from_numpy(draft).to(dev)
        acc_a = torch.full((R,), -1, dtype=torch.int32, device=dev)
        nxt_a = torch.full((R,), -1, dtype=torch.int32, device=dev)
        acc_b = torch.full((R,), -2, dtype=torch.int32, device=dev)
        nxt_b = torch.full((R,), -2, dtype=torch.int32, device=dev)

        st = L.w12_verify_greedy_noalloc(_ptr(lg_d), code, R, T, V, _ptr(dr_d), _ptr(acc_a),
                                         _ptr(nxt_a), stream)
        assert st == w12mod.OK, w12mod.status_string(st)
        nbytes = L.w12_verify_workspace_size(R, T, V)
        ws = w12mod.workspace(nbytes, dev)
        st = L.w12_verify_greedy(_ptr(lg_d), code, R, T, V, _ptr(dr_d), _ptr(acc_b), _ptr(nxt_b),
                                 _ptr(ws), nbytes, stream)
        assert st == w12mod.OK, w12mod.status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(acc_a, acc_b) and torch.equal(nxt_a, nxt_b)
        want = oracle.verify_greedy(lg, R, T, draft)
        assert acc_a.cpu().numpy().tolist() == want[0].tolist()
        assert nxt_a.cpu().numpy().tolist() == want[1].tolist()


def test_noalloc_rejects_oversized_problem(dev, w12mod):
    """A problem whose scratch would not fit the fixed array is refused
    before anything is launched."""
    import torch
    L = w12mod.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    R, T, V = 40000, 1, 8  # 40000 rows need more than the fixed scratch
    lg = torch.zeros((R * T, V), dtype=torch.float32, device=dev)
    acc = torch.zeros(R, dtype=torch.int32, device=dev)
    nxt = torch.zeros(R, dtype=torch.int32, device=dev)
    st = L.w12_verify_greedy_noalloc(_ptr(lg), w12mod.F32, R, T, V, None, _ptr(acc), _ptr(nxt),
                                     stream)
    assert st == w12mod.ERR_WORKSPACE
