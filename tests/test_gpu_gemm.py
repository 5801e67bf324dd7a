"""W12 decode-GEMM on the GPU against the oracle's fp64 product.

Acceptance (element by element): |y - y_ref| <= 2e-3 * sum_k |x_k w_k| + 1e-6
for fp32 y; bf16 y adds 2^-8 |y_ref|.  One-hot activations must reproduce a
weight row exactly: that pins the in-register rebuild and the escape patch
bit for bit inside the GEMM (SpecPilot repository page, "项目介绍": decoded
bit-exactly inside the GEMM).
"""
import numpy as np
import pytest

from helpers import bf16_bits_to_f64, check_gemm, dev_bits_to_np, ref_gemm_f64, to_dev_bits
from lossless_bit_weight_w12_gb300 import synth

pytestmark = pytest.mark.gpu


def _run(w12mod, dev, d, blob_d, x, path, y_dtype="f32"):
    import torch
    M = x.shape[0]
    x_d = to_dev_bits(x, dev)
    y_d = torch.empty((M, d.N), dtype=torch.float32 if y_dtype == "f32" else torch.bfloat16,
                      device=dev)
    ws = w12mod.workspace(w12mod.gemm_workspace_size(d, M), dev)
    w12mod.gemm(d, blob_d, x_d, y_d, ws, path=path)
    torch.cuda.synchronize()
    assert w12mod.get_device_error(ws) == 0
    if y_dtype == "f32":
        return y_d.cpu().numpy().astype(np.float64)
    return bf16_bits_to_f64(dev_bits_to_np(y_d))


def _paths(M):
    """Every explicit path that serves M: GEMV (M <= 4), mma.sync, tcgen05."""
    return [1, 2, 3] if M <= 4 else [2, 3]


SHAPES = [(128, 1), (128, 7), (384, 33), (1024, 130), (1152, 257), (5120, 96), (6144, 64)]
MS = [1, 2, 3, 4, 5, 8, 9, 16, 17, 32, 33, 64, 100, 128]


@pytest.mark.parametrize("K,N", SHAPES)
@pytest.mark.parametrize("M", MS)
def test_gemm_random_vs_oracle(dev, w12mod, oracle, K, N, M):
    rng = synth.streams(1000 + K + N + M, 2)
    w = synth.weights(rng[0], K, N)
    x = synth.activations(rng[1], M, K)
    d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
    od, oblob = oracle.encode(w, oracle.LAYOUT_NK)
    y_ref, s_ref = oracle.gemm(od, oblob, x)
    blob_d = w12mod.upload(blob, dev)
    for path in _paths(M):
        y = _run(w12mod, dev, d, blob_d, x, path)
        check_gemm(y, y_ref, s_ref, what=f"K={K} N={N} M={M} path={path}")


@pytest.mark.parametrize("M", [1, 3, 16, 40])
def test_gemm_bf16_output(dev, w12mod, oracle, M):
    K, N = 1024, 200
    rng = synth.streams(77 + M, 2)
    w = synth.weights(rng[0], K, N)
    x = synth.activations(rng[1], M, K)
    d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
    y_ref, s_ref = oracle.gemm(*oracle.encode(w, oracle.LAYOUT_NK), x)
    blob_d = w12mod.upload(blob, dev)
    for path in _paths(M):
        y = _run(w12mod, dev, d, blob_d, x, path, "bf16")
        check_gemm(y, y_ref, s_ref, bf16=True, what=f"bf16 M={M} path={path}")


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32, 128])
def test_gemm_one_hot_is_exact(dev, w12mod, M):
    """x = one-hot rows: y must equal the selected weight rows bit for bit,
    escapes included (the recipe plants zeros and subnormals, and this matrix
    adds NaN payloads and Infs)."""
    K, N = 2048, 300
    rng = synth.streams(5 + M, 2)
    w = synth.weights(rng[0], K, N)
    w[::7, 3] = 0x7FC1   # NaN payload rows in column 3 (escapes)
    w[5, ::11] = 0xFF80  # -Inf in row 5 (escapes)
    d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
    blob_d = w12mod.upload(blob, dev)
    ks = rng[1].integers(0, K, M)
    x = np.zeros((M, K), dtype=np.uint16)
    x[np.arange(M), ks] = 0x3F80
    want = bf16_bits_to_f64(w[:, ks].T)  # [M, N]
    # IEEE: the zero terms still turn an Inf or NaN weight elsewhere in the column into NaN
    nonfinite = ~np.isfinite(bf16_bits_to_f64(w))  # [N, K]
    for m, k in enumerate(ks):
        other = nonfinite.copy()
        other[:, k] = False
        want[m, other.any(axis=1)] = np.nan
    for path in _paths(M):
        y = _run(w12mod, dev, d, blob_d, x, path)
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(y), nan)
        np.testing.assert_array_equal(y[~nan], want[~nan])


def test_gemm_nonfinite(dev, w12mod, oracle):
    K, N, M = 512, 40, 3
    rng = synth.streams(9, 2)
    w = synth.weights(rng[0], K, N)
    w[3, 10] = 0x7F80  # +Inf   (w is [N, K])
    w[7, 200] = 0x7FC0  # NaN
    w[9, 300] = 0xFF80  # -Inf
    x = synth.activations(rng[1], M, K)
    x[:, :] = np.where(x == 0, 0x3F80, x)  # no zero activations (0 * Inf = NaN)
    d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
    y_ref, s_ref = oracle.gemm(*oracle.encode(w, oracle.LAYOUT_NK), x)
    blob_d = w12mod.upload(blob, dev)
    for path in _paths(M):
        y = _run(w12mod, dev, d, blob_d, x, path)
        check_gemm(y, y_ref, s_ref, what=f"nonfinite path={path}")


@pytest.mark.parametrize("path,M", [(2, 16), (3, 16), (3, 64), (3, 128)])
def test_gemm_deterministic(dev, w12mod, path, M):
    """Stream-K partial sums are added in a fixed order: repeated calls give
    the same bits (K = 17408 spreads every column tile over several CTAs;
    the tcgen05 rings are even at M = 16 and 64, odd at M = 128)."""
    import torch
    K, N = 17408, 640
    rng = synth.streams(3, 2)
    w = synth.weights(rng[0], K, N)
    x = to_dev_bits(synth.activations(rng[1], M, K), dev)
    d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
    blob_d = w12mod.upload(blob, dev)
    ws = w12mod.workspace(w12mod.gemm_workspace_size(d, M), dev)
    ys = []
    for _ in range(3):
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        w12mod.gemm(d, blob_d, x, y, ws, path=path)
        ys.append(y)
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[1], ys[2])


FULL_MS = (1, 16, 32, 64, 128)


def _layer_inputs(seed, Ms):
    """The layer's six weights (stream i) and, per M, their activations."""
    rng = synth.streams(seed, len(synth.LAYER_SHAPES) + 8)
    ws = [synth.weights(rng[i], K, N) for i, (_, K, N) in enumerate(synth.LAYER_SHAPES)]
    xs = {M: [synth.activations(synth.streams(seed * 1000 + M, len(synth.LAYER_SHAPES))[i], M, K)
              for i, (_, K, _) in enumerate(synth.LAYER_SHAPES)] for M in Ms}
    return ws, xs


@pytest.mark.parametrize("seed", [1, 3])
def test_gemm_full_layer_every_output(dev, w12mod, oracle, seed):
    """Config-1..3 layer shapes at full size, one GEMM launch per matrix as
    w12_gemm plans it, at M = 1, 16, 32, 64, 128 on the AUTO path and every
    path that serves M: every output against the float64 definition, and 24
    sampled columns against the oracle itself."""
    ws, xs = _layer_inputs(seed, FULL_MS)
    for i, (name, K, N) in enumerate(synth.LAYER_SHAPES):
        w = ws[i]
        d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
        blob_d = w12mod.upload(blob, dev)
        refs = dict(zip(FULL_MS, ref_gemm_f64(w, [xs[M][i] for M in FULL_MS])))
        ns = np.unique(np.r_[np.random.default_rng(i).integers(0, N, 22), [0, N - 1]])
        od, oblob = oracle.encode(w[ns], oracle.LAYOUT_NK)
        for M in FULL_MS:
            y_ref, s_ref = refs[M]
            yo_ref, so_ref = oracle.gemm(od, oblob, xs[M][i])
            for path in [0] + _paths(M):
                y = _run(w12mod, dev, d, blob_d, xs[M][i], path)
                check_gemm(y, y_ref, s_ref, what=f"{name} M={M} path={path} (every output)")
                check_gemm(y[:, ns], yo_ref, so_ref, what=f"{name} M={M} path={path} (oracle)")
        del blob_d


def test_gemm_argument_errors(dev, w12mod):
    import torch
    K, N = 256, 16
    w = np.full((N, K), 0x3F80, dtype=np.uint16)
    d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
    blob_d = w12mod.upload(blob, dev)
    x = torch.zeros((4, K), dtype=torch.int16, device=dev)
    y = torch.empty((4, N), dtype=torch.float32, device=dev)
    need = w12mod.gemm_workspace_size(d, 4)
    assert need >= 256
    small = w12mod.workspace(256, dev)[:128]
    with pytest.raises(w12mod.W12Error) as e:
        w12mod.gemm(d, blob_d, x, y, small)
    assert e.value.status == w12mod.ERR_WORKSPACE
    ws = w12mod.workspace(need, dev)
    with pytest.raises(w12mod.W12Error) as e:  # the GEMV path serves M <= 4 only
        w12mod.gemm(d, blob_d, torch.zeros((5, K), dtype=torch.int16, device=dev),
                    torch.empty((5, N), dtype=torch.float32, device=dev), ws,
                    path=w12mod.PATH_GEMV)
    assert e.value.status == w12mod.ERR_SHAPE
    with pytest.raises(w12mod.W12Error) as e:
        w12mod.gemm(d, blob_d, torch.zeros((129, K), dtype=torch.int16, device=dev),
                    torch.empty((129, N), dtype=torch.float32, device=dev), ws)
    assert e.value.status == w12mod.ERR_SHAPE
    xs = torch.zeros(4 * K + 8, dtype=torch.int16, device=dev)[1:1 + 4 * K].view(4, K)
    with pytest.raises(w12mod.W12Error) as e:
        w12mod.gemm(d, blob_d, xs, y, ws)
    assert e.value.status == w12mod.ERR_ALIGN


def test_gemm_k_zero_writes_zeros(dev, w12mod):
    import torch
    w = np.zeros((9, 0), dtype=np.uint16)
    d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
    y = torch.full((2, 9), 5.0, dtype=torch.float32, device=dev)
    x = torch.zeros((2, 0), dtype=torch.int16, device=dev)
    ws = w12mod.workspace(256, dev)
    w12mod.gemm(d, w12mod.workspace(256, dev), x, y, ws)
    assert torch.count_nonzero(y).item() == 0


def _batched(w12mod, dev, items, M, y_dtype="f32", path=0):
    """items: list of (desc, blob_dev, x uint16 [M,K]); returns list of fp64 y."""
    import torch
    xs = [to_dev_bits(x, dev) for _, _, x in items]
    ys = [torch.empty((M, d.N), dtype=torch.float32 if y_dtype == "f32" else torch.bfloat16, device=dev)
          for d, _, _ in items]
    descs = [d for d, _, _ in items]
    ws = w12mod.workspace(w12mod.gemm_batched_workspace_size(descs, M), dev)
    w12mod.gemm_batched(descs, [b for _, b, _ in items], xs, ys, ws, path=path)
    torch.cuda.synchronize()
    assert w12mod.get_device_error(ws) == 0
    if y_dtype == "f32":
        return [y.cpu().numpy().astype(np.float64) for y in ys]
    return [bf16_bits_to_f64(dev_bits_to_np(y)) for y in ys]


@pytest.mark.parametrize("M", [1, 2, 3, 4, 16, 33, 128])
def test_gemm_batched_mixed_shapes(dev, w12mod, oracle, M):
    """One launch over products of different K and N (ragged tiles and unit
    counts), each checked against the oracle."""
    shapes = [(384, 33), (1024, 130), (128, 7), (1152, 257), (2048, 16)]
    rng = synth.streams(4000 + M, 2 * len(shapes))
    items, refs = [], []
    for i, (K, N) in enumerate(shapes):
        w = synth.weights(rng[2 * i], K, N)
        x = synth.activations(rng[2 * i + 1], M, K)
        d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
        items.append((d, w12mod.upload(blob, dev), x))
        refs.append(oracle.gemm(*oracle.encode(w, oracle.LAYOUT_NK), x))
    for path in _paths(M):
        for rep in range(2):  # the workspace is reused by the second call
            ys = _batched(w12mod, dev, items, M, path=path)
            for (K, N), y, (y_ref, s_ref) in zip(shapes, ys, refs):
                check_gemm(y, y_ref, s_ref, what=f"batched K={K} N={N} M={M} path={path}")


@pytest.mark.parametrize("M,path", [(2, 1), (16, 2), (16, 3), (100, 3)])
def test_gemm_batched_repeatable(dev, w12mod, M, path):
    """Repeated batched calls give the same bits: partial sums are combined
    in unit order, whichever CTA finishes a tile."""
    shapes = [(5120, 1030), (17408, 300), (384, 33)]
    rng = synth.streams(4100 + M, 2 * len(shapes))
    items = []
    for i, (K, N) in enumerate(shapes):
        d, blob = w12mod.encode(synth.weights(rng[2 * i], K, N), w12mod.LAYOUT_NK)
        items.append((d, w12mod.upload(blob, dev), synth.activations(rng[2 * i + 1], M, K)))
    ya = _batched(w12mod, dev, items, M, path=path)
    yb = _batched(w12mod, dev, items, M, path=path)
    for a, bb in zip(ya, yb):
        assert np.array_equal(a, bb)


def test_gemm_batched_full_layer(dev, w12mod, oracle):
    """The layer's six linears in one launch (the launch the bench times),
    full size, M = 1, 4, 16, 32, 64, 128 on the AUTO path and every path that
    serves M: every output against the float64 definition, sampled columns
    against the oracle."""
    Ms = (1, 4, 16, 32, 64, 128)
    ws, xs = _layer_inputs(1, Ms)
    items = {M: [] for M in Ms}
    refs = {M: [] for M in Ms}
    orefs = {M: [] for M in Ms}
    blobs = []
    for i, (name, K, N) in enumerate(synth.LAYER_SHAPES):
        d, blob = w12mod.encode(ws[i], w12mod.LAYOUT_NK)
        blobs.append((d, w12mod.upload(blob, dev)))
        for M, r in zip(Ms, ref_gemm_f64(ws[i], [xs[M][i] for M in Ms])):
            refs[M].append(r)
        ns = np.unique(np.r_[np.random.default_rng(i).integers(0, N, 20), [0, N - 1]])
        od, oblob = oracle.encode(ws[i][ns], oracle.LAYOUT_NK)
        for M in Ms:
            orefs[M].append((ns, oracle.gemm(od, oblob, xs[M][i])))
    for M in Ms:
        items = [(d, b, xs[M][i]) for i, (d, b) in enumerate(blobs)]
        for path in [0] + _paths(M):
            ys = _batched(w12mod, dev, items, M, path=path)
            for i, (name, K, N) in enumerate(synth.LAYER_SHAPES):
                y_ref, s_ref = refs[M][i]
                check_gemm(ys[i], y_ref, s_ref, what=f"batched {name} M={M} path={path} (every output)")
                ns, (yo, so) = orefs[M][i]
                check_gemm(ys[i][:, ns], yo, so, what=f"batched {name} M={M} path={path} (oracle)")


@pytest.mark.parametrize("M", [1, 4, 16, 33, 64, 128])
def test_gemm_early_weights_option(dev, w12mod, oracle, M):
    """W12_OPT_EARLY_WEIGHTS (the weight stream starts under the previous
    kernel's tail; the launch configuration the bench times) gives the same
    bits as the default launch on every path, single and batched, on blobs
    uploaded before the calls."""
    import torch
    shapes = [(1024, 130), (2048, 257), (384, 33)]
    rng = synth.streams(4200 + M, 2 * len(shapes))
    items, refs = [], []
    for i, (K, N) in enumerate(shapes):
        w = synth.weights(rng[2 * i], K, N)
        x = synth.activations(rng[2 * i + 1], M, K)
        d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
        items.append((d, w12mod.upload(blob, dev), x))
        refs.append(oracle.gemm(*oracle.encode(w, oracle.LAYOUT_NK), x))
    torch.cuda.synchronize()
    for path in [0] + _paths(M):
        ys_default = _batched(w12mod, dev, items, M, path=path)
        ys_early = _batched(w12mod, dev, items, M, path=path | w12mod.OPT_EARLY_WEIGHTS)
        for (K, N), a, e, (y_ref, s_ref) in zip(shapes, ys_default, ys_early, refs):
            assert np.array_equal(a, e), f"early weights changed the result K={K} N={N} M={M} path={path}"
            check_gemm(e, y_ref, s_ref, what=f"early weights K={K} N={N} M={M} path={path}")
        for (d, b, x), (y_ref, s_ref) in zip(items, refs):
            y = _run(w12mod, dev, d, b, x, path | w12mod.OPT_EARLY_WEIGHTS)
            check_gemm(y, y_ref, s_ref, what=f"early weights single M={M} path={path}")


def test_gemm_batched_argument_errors(dev, w12mod):
    import torch
    w = np.full((16, 256), 0x3F80, dtype=np.uint16)
    d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
    b = w12mod.upload(blob, dev)
    x = torch.zeros((1, 256), dtype=torch.int16, device=dev)
    y = torch.empty((1, 16), dtype=torch.float32, device=dev)
    assert w12mod.gemm_batched_workspace_size([d] * 9, 1) == 0  # more than W12_MAX_BATCH
    need = w12mod.gemm_batched_workspace_size([d, d], 1)
    with pytest.raises(w12mod.W12Error) as e:
        w12mod.gemm_batched([d, d], [b, b], [x, x], [y, y], w12mod.workspace(256, dev)[:64])
    assert e.value.status == w12mod.ERR_WORKSPACE
    w12mod.gemm_batched([d, d], [b, b], [x, x], [y, y], w12mod.workspace(need, dev))
