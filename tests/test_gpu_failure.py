"""Failure detection on the GPU without a GPU fault, and the safe default of
programmatic dependent launch.

- Bounded waits: w12_gemm_batched_debug withholds one unit's weight copy, so
  a full barrier is never completed; with a 20 ms wait limit every kernel
  still runs to its end, the workspace reads W12_ERR_TIMEOUT, and the next
  normal call on the same workspace matches the oracle.
- Device-detected blob errors: an escape range past the escape list is not
  followed by the GEMM kernels (GEMV, mma.sync, tcgen05) nor by the fused
  lm_head verify; the workspace reads W12_ERR_DEVICE and the context stays
  usable.
- A blob written by the kernel launched just before a GEMM on the same
  stream (the device encoder, a torch kernel) is read after that kernel
  completed: by default the GEMM reads nothing before griddepcontrol.wait.
"""
import numpy as np
import pytest

from helpers import check_gemm, to_dev_bits
from lossless_bit_weight_w12_gb300 import synth

pytestmark = pytest.mark.gpu

# (path, M): the GEMV, mma.sync and tcgen05 consumers
PATHS = [(1, 1), (2, 16), (3, 64), (3, 128)]


def _batch(w12mod, oracle, dev, M, seed):
    """Two products (one with an odd tile count), the oracle's results."""
    import torch
    rng = synth.streams(seed, 4)
    shapes = [(1024, 640), (2048, 392)]
    descs, blobs, xs, ys, refs = [], [], [], [], []
    for i, (K, N) in enumerate(shapes):
        w = synth.weights(rng[2 * i], K, N)
        x = synth.activations(rng[2 * i + 1], M, K)
        d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
        descs.append(d)
        blobs.append(w12mod.upload(blob, dev))
        xs.append(to_dev_bits(x, dev))
        ys.append(torch.empty((M, N), dtype=torch.float32, device=dev))
        refs.append(oracle.gemm(*oracle.encode(w, oracle.LAYOUT_NK), x))
    return descs, blobs, xs, ys, refs


@pytest.mark.parametrize("path,M", PATHS)
def test_withheld_copy_times_out_and_the_next_call_is_correct(dev, w12mod, oracle, path, M):
    import torch
    descs, blobs, xs, ys, refs = _batch(w12mod, oracle, dev, M, 70 + M)
    ws = w12mod.workspace(w12mod.gemm_batched_workspace_size(descs, M), dev)
    for unit in (3, 17):
        w12mod.gemm_batched_debug(descs, blobs, xs, ys, ws, withhold_unit=unit, wait_limit_us=20000, path=path)
        torch.cuda.synchronize()
        assert w12mod.get_device_error(ws) == w12mod.ERR_TIMEOUT
        # the same workspace, no clearing: counters were left at zero
        w12mod.gemm_batched(descs, blobs, xs, ys, ws, path=path)
        torch.cuda.synchronize()
        assert w12mod.get_device_error(ws) == 0
        for y, (y_ref, s_ref) in zip(ys, refs):
            check_gemm(y.cpu().numpy().astype(np.float64), y_ref, s_ref, what=f"after timeout path={path}")


@pytest.mark.parametrize("path,M", PATHS)
def test_debug_call_without_hooks_is_the_plain_call(dev, w12mod, oracle, path, M):
    import torch
    descs, blobs, xs, ys, refs = _batch(w12mod, oracle, dev, M, 90 + M)
    ws = w12mod.workspace(w12mod.gemm_batched_workspace_size(descs, M), dev)
    w12mod.gemm_batched_debug(descs, blobs, xs, ys, ws, withhold_unit=-1, wait_limit_us=0, path=path)
    torch.cuda.synchronize()
    assert w12mod.get_device_error(ws) == 0
    for y, (y_ref, s_ref) in zip(ys, refs):
        check_gemm(y.cpu().numpy().astype(np.float64), y_ref, s_ref, what=f"debug path={path}")


def _corrupt(blob):
    """Column 1's escape range of unit 0 now ends past the escape list."""
    bad = blob.copy()
    meta = bad[3 * 8192:3 * 8192 + 4 * 129].view(np.uint32)
    meta[2] = (meta[2] & 0xFF) | (100000 << 8)
    return bad


@pytest.mark.parametrize("path,M", PATHS)
def test_gemm_corrupt_escape_range_is_contained(dev, w12mod, oracle, path, M):
    import torch
    K, N = 1024, 384
    rng = synth.streams(31, 2)
    w = synth.weights(rng[0], K, N)
    w[1, 5] = 0x0000  # an escape in column 1
    x = synth.activations(rng[1], M, K)
    d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
    x_d = to_dev_bits(x, dev)
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    ws = w12mod.workspace(w12mod.gemm_workspace_size(d, M), dev)
    w12mod.gemm(d, w12mod.upload(_corrupt(blob), dev), x_d, y, ws, path=path)
    torch.cuda.synchronize()
    assert w12mod.get_device_error(ws) == w12mod.ERR_DEVICE
    # the context and the workspace stay usable
    w12mod.gemm(d, w12mod.upload(blob, dev), x_d, y, ws, path=path)
    torch.cuda.synchronize()
    assert w12mod.get_device_error(ws) == 0
    y_ref, s_ref = oracle.gemm(*oracle.encode(w, oracle.LAYOUT_NK), x)
    check_gemm(y.cpu().numpy().astype(np.float64), y_ref, s_ref, what=f"after corrupt path={path}")


@pytest.mark.parametrize("R,T", [(1, 1), (4, 16)])  # mma.sync and tcgen05 fused kernels
def test_lmhead_verify_corrupt_escape_range_is_contained(dev, w12mod, oracle, R, T):
    import torch
    K, N = 1024, 1000
    rng = synth.streams(41 + R, 3)
    w = synth.weights(rng[0], K, N)
    w[1, 5] = 0x0000
    hid = synth.activations(rng[1], R * T, K)
    d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
    draft = torch.from_numpy(rng[2].integers(0, N, (R, T - 1)).astype(np.int32)).to(dev)
    acc = torch.empty(R, dtype=torch.int32, device=dev)
    nxt = torch.empty(R, dtype=torch.int32, device=dev)
    lg = torch.empty((R * T, N), dtype=torch.float32, device=dev)
    ws = w12mod.workspace(w12mod.verify_lmhead_workspace_size(d, R, T), dev)
    hid_d = to_dev_bits(hid, dev)
    w12mod.verify_greedy_lmhead(hid_d, d, w12mod.upload(_corrupt(blob), dev), R, T, draft, acc, nxt, ws,
                                logits_out_dev=lg)
    torch.cuda.synchronize()
    assert w12mod.get_device_error(ws) == w12mod.ERR_DEVICE
    w12mod.verify_greedy_lmhead(hid_d, d, w12mod.upload(blob, dev), R, T, draft, acc, nxt, ws,
                                logits_out_dev=lg)
    torch.cuda.synchronize()
    assert w12mod.get_device_error(ws) == 0
    want = oracle.verify_greedy(lg.cpu().numpy(), R, T, draft.cpu().numpy())
    assert acc.cpu().numpy().tolist() == want[0].tolist()
    assert nxt.cpu().numpy().tolist() == want[1].tolist()


@pytest.mark.parametrize("path,M", PATHS)
def test_blob_written_by_the_previous_kernel(dev, w12mod, oracle, path, M):
    """The device encoder, then at once the GEMM on the same stream; and a
    torch kernel writing the blob, then at once the GEMM (default launch:
    no weight read before the previous kernel completed)."""
    import torch
    K, N = 2048, 520
    rng = synth.streams(51 + M, 2)
    w = synth.weights(rng[0], K, N)
    x = synth.activations(rng[1], M, K)
    y_ref, s_ref = oracle.gemm(*oracle.encode(w, oracle.LAYOUT_NK), x)
    x_d = to_dev_bits(x, dev)
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    w_d = to_dev_bits(w, dev)
    torch.cuda.synchronize()
    d, blob_d = w12mod.encode_device(w_d)
    ws = w12mod.workspace(w12mod.gemm_workspace_size(d, M), dev)
    w12mod.gemm(d, blob_d, x_d, y, ws, path=path)
    torch.cuda.synchronize()
    assert w12mod.get_device_error(ws) == 0
    check_gemm(y.cpu().numpy().astype(np.float64), y_ref, s_ref, what=f"after encode_device path={path}")
    # a fresh blob buffer written by a torch elementwise kernel, GEMM right after
    for trial in range(3):
        dst = torch.empty(blob_d.numel() + 256, dtype=torch.uint8, device=dev)
        off = (-dst.data_ptr()) % 256
        dst = dst[off:off + blob_d.numel()]
        dst.fill_(0xA5)
        torch.cuda.synchronize()
        torch.bitwise_or(blob_d, 0, out=dst)
        w12mod.gemm(d, dst, x_d, y, ws, path=path)
        torch.cuda.synchronize()
        assert w12mod.get_device_error(ws) == 0
        check_gemm(y.cpu().numpy().astype(np.float64), y_ref, s_ref, what=f"torch-written blob {trial}")
