"""Pins of the oracle's fp64 GEMM and greedy verification.

GEMM (y[m,n] = sum_k x[m,k] w[k,n]):
- one-hot rows of x pick out one row of W exactly (a transposed operand, a
  wrong index or a dropped escape fails this on a non-square shape);
- small-integer operands make every partial sum exact in fp64, so the result
  must equal Python's exact integer arithmetic;
- random operands agree with numpy's float64 matmul of the ORIGINAL weights
  (not the oracle's decode) up to fp64 rounding-order error;
- the sampled-output entry returns the same values as the full product.

Verify (SpecPilot summary p5 "Risks" bullet 3: every committed token is the
target's greedy choice; p4 "结果与验证": token-by-token check):
- hand cases: all-equal rows, full accept, immediate reject, NaN, -0/+0;
- argmax equals numpy.argmax (first maximum, first NaN) on random rows with
  forced ties.
"""
import numpy as np
import pytest

from lossless_bit_weight_w12_gb300 import synth


def _f64(bits):
    return synth.bf16_to_f32(bits).astype(np.float64)


@pytest.mark.parametrize("layout", [0, 1])
def test_gemm_one_hot(oracle, layout):
    rng = synth.streams(11, 1)[0]
    K, N = 384, 40
    w_nk = synth.weights(rng, K, N)
    w_kn = np.ascontiguousarray(w_nk.T)
    d, blob = oracle.encode(w_kn if layout == 0 else w_nk, layout)
    ks = [0, 1, 7, 128, 255, 383]
    x = np.zeros((len(ks), K), dtype=np.uint16)
    for m, k in enumerate(ks):
        x[m, k] = 0x3F80  # 1.0
    y, s = oracle.gemm(d, blob, x)
    for m, k in enumerate(ks):
        np.testing.assert_array_equal(y[m], _f64(w_kn[k]))
        np.testing.assert_array_equal(s[m], np.abs(_f64(w_kn[k])))


def test_gemm_exact_integers(oracle):
    rng = np.random.default_rng(5)
    K, N, M = 256, 24, 3
    wi = rng.integers(-8, 9, size=(K, N))
    xi = rng.integers(-8, 9, size=(M, K))
    w = synth.bf16_rne(wi.astype(np.float32))
    x = synth.bf16_rne(xi.astype(np.float32))
    d, blob = oracle.encode(w, oracle.LAYOUT_KN)
    y, s = oracle.gemm(d, blob, x)
    want = [[sum(int(xi[m, k]) * int(wi[k, n]) for k in range(K)) for n in range(N)]
            for m in range(M)]
    np.testing.assert_array_equal(y, np.array(want, dtype=np.float64))
    np.testing.assert_array_equal(s, np.abs(xi).astype(np.float64) @ np.abs(wi).astype(np.float64))


def test_gemm_matches_numpy_float64(oracle):
    rng = synth.streams(12, 2)
    K, N, M = 640, 33, 5
    w_nk = synth.weights(rng[0], K, N)
    x = synth.activations(rng[1], M, K)
    d, blob = oracle.encode(w_nk, oracle.LAYOUT_NK)
    y, s = oracle.gemm(d, blob, x)
    ref = _f64(x) @ _f64(w_nk).T
    assert np.all(np.abs(y - ref) <= 1e-13 * s + 1e-300)
    # sampled outputs are the same numbers
    ms = np.array([0, 4, 2, 3])
    ns = np.array([0, 32, 17, 5])
    ys, ss = oracle.gemm_at(d, blob, x, ms, ns)
    np.testing.assert_array_equal(ys, y[ms, ns])
    np.testing.assert_array_equal(ss, s[ms, ns])


def test_gemm_nonfinite_classes(oracle):
    K, N = 128, 4
    w = np.full((K, N), 0x3F80, dtype=np.uint16)
    w[3, 1] = 0x7F80   # +Inf in column 1
    w[4, 2] = 0x7FC0   # NaN in column 2
    w[5, 3] = 0xFF80   # -Inf in column 3
    d, blob = oracle.encode(w, oracle.LAYOUT_KN)
    x = np.full((1, K), 0x3F80, dtype=np.uint16)
    y, _ = oracle.gemm(d, blob, x)
    assert y[0, 0] == 128.0
    assert y[0, 1] == np.inf
    assert np.isnan(y[0, 2])
    assert y[0, 3] == -np.inf


def test_verify_hand_cases(oracle):
    V, T = 10, 5
    # all-equal rows: argmax 0 everywhere
    lg = np.zeros((T, V), dtype=np.float32)
    acc, nxt = oracle.verify_greedy(lg, 1, T, np.zeros((1, T - 1), np.int32))
    assert acc[0] == T - 1 and nxt[0] == 0
    # full accept: drafts equal the argmaxes; next is the last row's argmax
    lg = np.zeros((T, V), dtype=np.float32)
    tgt = [3, 1, 4, 1, 5]
    for i, t in enumerate(tgt):
        lg[i, t] = 1.0
    acc, nxt = oracle.verify_greedy(lg, 1, T, np.array([tgt[:4]], np.int32))
    assert acc[0] == 4 and nxt[0] == 5
    # immediate reject
    acc, nxt = oracle.verify_greedy(lg, 1, T, np.array([[2, 1, 4, 1]], np.int32))
    assert acc[0] == 0 and nxt[0] == 3
    # reject in the middle
    acc, nxt = oracle.verify_greedy(lg, 1, T, np.array([[3, 1, 9, 1]], np.int32))
    assert acc[0] == 2 and nxt[0] == 4
    # T = 1: nothing to verify, next is row 0's argmax
    acc, nxt = oracle.verify_greedy(lg[:1], 1, 1, np.zeros((1, 0), np.int32))
    assert acc[0] == 0 and nxt[0] == 3


def test_argmax_special_values(oracle):
    row = np.array([[-0.0, 0.0, -1.0]], dtype=np.float32)
    assert oracle.argmax(row)[0] == 0              # -0 == +0: lowest index
    row = np.array([[0.0, -0.0, -1.0]], dtype=np.float32)
    assert oracle.argmax(row)[0] == 0
    row = np.array([[1.0, np.inf, np.nan, np.nan, 5.0]], dtype=np.float32)
    assert oracle.argmax(row)[0] == 2              # first NaN wins over +Inf
    row = np.array([[-np.inf, -np.inf]], dtype=np.float32)
    assert oracle.argmax(row)[0] == 0
    row = np.array([[3.0, 7.0, 7.0, 2.0]], dtype=np.float32)
    assert oracle.argmax(row)[0] == 1
    # bf16 logits: same rule on the widened values
    b = synth.bf16_rne(np.array([[1.0, 2.0, 2.0, np.nan]], dtype=np.float32))
    b[0, 3] = 0xFFC1  # negative-signed NaN is still NaN
    assert oracle.argmax(b)[0] == 3


@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_argmax_matches_numpy(oracle, dtype):
    rng = np.random.default_rng(9)
    rows, V = 64, 1000
    lg = synth.logits(rng, rows, V, dtype=dtype)
    f = synth.bf16_to_f32(lg) if dtype == np.uint16 else lg
    # force ties between the max and a later index, and plant NaNs in some rows
    for r in range(0, rows, 4):
        j = int(np.argmax(f[r]))
        t = int(rng.integers(0, V))
        lg[r, t] = lg[r, j]
    for r in range(1, rows, 8):
        lg[r, int(rng.integers(0, V))] = 0x7FC0 if dtype == np.uint16 else np.nan
    f = synth.bf16_to_f32(lg) if dtype == np.uint16 else lg
    np.testing.assert_array_equal(oracle.argmax(lg), np.argmax(f, axis=1))


def test_verify_matches_numpy_argmax(oracle):
    rng = np.random.default_rng(10)
    R, T, V = 6, 16, 5000
    lg = synth.logits(rng, R * T, V)
    g = np.argmax(lg, axis=1).reshape(R, T)
    d = synth.draft_tokens(rng, g, R, T, V)
    acc, nxt = oracle.verify_greedy(lg, R, T, d)
    for r in range(R):
        L = next((i for i in range(T - 1) if d[r, i] != g[r, i]), T - 1)
        assert acc[r] == L and nxt[r] == g[r, L]
