"""Shared helpers for the GPU parity tests (device buffers, tolerances)."""
import numpy as np

# fp32 GEMM acceptance: |y - y_ref| <= 2e-3 * sum_k |x w| + 1e-6
REL, ABS = 2e-3, 1e-6
# bf16 output adds half a bf16 ulp (2^-9 |y|); 2^-8 leaves margin for the fp32 sum
BF16_EXTRA = 2.0 ** -8


def to_dev_bits(a, dev):
    """uint16 bit patterns -> torch int16 on dev (the library reads them as bf16)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).to(dev)


def dev_bits_to_np(t):
    return t.cpu().contiguous().view(__import__("torch").int16).numpy().view(np.uint16)


def bf16_bits_to_f64(u):
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_gemm(y, y_ref, s_ref, bf16=False, what=""):
    """Element-wise acceptance with non-finite classes matched exactly."""
    y = np.asarray(y, dtype=np.float64)
    fin = np.isfinite(y_ref)
    assert np.array_equal(np.isnan(y), np.isnan(y_ref)), f"{what}: NaN pattern differs"
    inf = np.isinf(y_ref)
    assert np.array_equal(y[inf], y_ref[inf]), f"{what}: Inf values differ"
    tol = REL * s_ref + ABS
    if bf16:
        tol = tol + BF16_EXTRA * np.abs(y_ref)
    err = np.abs(y - y_ref)
    bad = fin & ~(err <= tol)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} outputs outside tolerance; first {tuple(i)}: "
            f"y={y[tuple(i)]!r} ref={y_ref[tuple(i)]!r} tol={tol[tuple(i)]!r}")


def ref_gemm_f64(w, xs, chunk=4096):
    """The GEMM's definition on the uncompressed weights: y = x . W summed in
    float64 (a product of two bf16 values is exact in float64), and the
    tolerance scale S = |x| . |W|.  w: bf16 bits [N, K]; xs: a list of bf16
    bits [M_i, K].  Returns [(y_ref, s_ref)] per x, [M_i, N] each.  Column
    chunks bound the float64 copy of W.  This is the definition the oracle's
    GEMM is pinned to (tests/test_oracle_gemm_verify.py), applied to every
    output of a full-size matrix where the oracle itself would take minutes."""
    N, K = w.shape
    xa = np.concatenate([bf16_bits_to_f64(x) for x in xs], axis=0)
    ya = np.empty((xa.shape[0], N), dtype=np.float64)
    sa = np.empty((xa.shape[0], N), dtype=np.float64)
    xabs = np.abs(xa)
    for c0 in range(0, N, chunk):
        wf = bf16_bits_to_f64(w[c0:c0 + chunk])
        ya[:, c0:c0 + chunk] = xa @ wf.T
        sa[:, c0:c0 + chunk] = xabs @ np.abs(wf).T
    out, r = [], 0
    for x in xs:
        out.append((ya[r:r + x.shape[0]], sa[r:r + x.shape[0]]))
        r += x.shape[0]
    return out
