"""GPU decode (blob -> bf16) against the input weights: bit-exact.

The format is lossless (SpecPilot summary, airadar.tv English edition,
"Reasons" bullet 2), so decode(encode(W)) must return W's exact bit patterns,
including +-0, subnormals, Inf, NaN payloads and escaped exponents.
"""
import numpy as np
import pytest

from helpers import dev_bits_to_np
from lossless_bit_weight_w12_gb300 import synth

pytestmark = pytest.mark.gpu


def _cases():
    rng = synth.streams(31, 6)
    allp = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    yield "recipe", synth.weights(rng[0], 1024, 1024)
    yield "recipe_ragged", synth.weights(rng[1], 384, 131)
    yield "random_bits", synth.random_bits(rng[2], (77, 640))
    yield "all_patterns", np.random.default_rng(2).permutation(allp).reshape(64, 1024)
    yield "all_patterns_ordered", allp.reshape(512, 128)
    yield "one_column", synth.weights(rng[3], 5120, 1)
    yield "one_group", synth.weights(rng[4], 128, 1)


CASES = list(_cases())


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("layout", [0, 1], ids=["out_KN", "out_NK"])
def test_decode_bit_exact(dev, w12mod, oracle, name, w, layout):
    import torch
    d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
    blob_d = w12mod.upload(blob, dev)
    N, K = w.shape
    shape = (K, N) if layout == w12mod.LAYOUT_KN else (N, K)
    out = torch.full(shape, -1, dtype=torch.int16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    w12mod.decode(d, blob_d, out, layout, err)
    got = dev_bits_to_np(out)
    want = w.T if layout == w12mod.LAYOUT_KN else w
    np.testing.assert_array_equal(got, want)
    assert int(err.item()) == 0


def test_decode_full_layer_shapes(dev, w12mod):
    """Every config-1 layer matrix at full size (q, k, v, o, gate_up, down)."""
    import torch
    rng = synth.streams(1, len(synth.LAYER_SHAPES))
    for i, (name, K, N) in enumerate(synth.LAYER_SHAPES):
        w = synth.weights(rng[i], K, N)
        d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
        blob_d = w12mod.upload(blob, dev)
        out = torch.empty((N, K), dtype=torch.int16, device=dev)
        w12mod.decode(d, blob_d, out, w12mod.LAYOUT_NK)
        ref = torch.from_numpy(w.view(np.int16)).to(dev)
        assert torch.equal(out, ref), name
        del out, ref, blob_d


def test_decode_corrupt_escape_range_is_contained(dev, w12mod):
    """A meta word pointing past the escape list is not followed: the kernel
    records W12_ERR_DEVICE and finishes."""
    import torch
    w = np.full((4, 128), 0x3F80, dtype=np.uint16)
    w[1, 5] = 0x0000  # one escape, in column 1 (the only unit block)
    d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
    bad = blob.copy()
    meta = bad[3 * 8192:3 * 8192 + 4 * 129].view(np.uint32)  # the unit's meta words
    meta[2] = (meta[2] & 0xFF) | (1000 << 8)  # column 1's range now ends at 1000
    blob_d = w12mod.upload(bad, dev)
    out = torch.empty((4, 128), dtype=torch.int16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    w12mod.decode(d, blob_d, out, w12mod.LAYOUT_NK, err)
    torch.cuda.synchronize()
    assert int(err.item()) == w12mod.ERR_DEVICE


def test_decode_argument_errors(dev, w12mod):
    import torch
    w = np.full((2, 128), 0x3F80, dtype=np.uint16)
    d, blob = w12mod.encode(w, w12mod.LAYOUT_NK)
    blob_d = w12mod.upload(blob, dev)
    out = torch.empty((2, 128), dtype=torch.int16, device=dev)
    with pytest.raises(w12mod.W12Error) as e:
        w12mod.decode(d, blob_d[1:], out)  # not 256-byte aligned
    assert e.value.status == w12mod.ERR_ALIGN
    from dataclasses import replace
    with pytest.raises(w12mod.W12Error) as e:
        w12mod.decode(replace(d, off_esc=d.off_esc + 256), blob_d, out)
    assert e.value.status == w12mod.ERR_BLOB
