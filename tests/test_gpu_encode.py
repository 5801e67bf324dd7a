"""GPU encoder (w12_encode_plan_device / w12_encode_device) against the
oracle: the same descriptor and the same blob, byte for byte.

The encoder is the setup side of the lossless W12 format (SpecPilot summary,
airadar.tv English edition, "Reasons" bullet 2: BF16 split into three 4-bit
planes); a blob the device writes must be the one the written format (and so
the oracle's encoder) defines, for every bf16 pattern, both input
orientations, ragged column counts and the layer's full-size shapes.
"""
import numpy as np
import pytest

from lossless_bit_weight_w12_gb300 import synth

pytestmark = pytest.mark.gpu


def _cases():
    rng = synth.streams(41, 6)
    allp = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    yield "recipe_nk", synth.weights(rng[0], 1024, 300), 1
    yield "recipe_kn", np.ascontiguousarray(synth.weights(rng[1], 512, 131).T), 0
    yield "random_bits", synth.random_bits(rng[2], (77, 640)), 1
    yield "all_patterns", np.random.default_rng(3).permutation(allp).reshape(64, 1024), 1
    yield "all_patterns_ordered_kn", allp.reshape(512, 128), 0
    yield "one_group", synth.weights(rng[3], 128, 1), 1
    yield "q_full", synth.weights(rng[4], 5120, 6144), 1


CASES = list(_cases())


def _to_dev(w, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(w).view(np.int16)).to(dev)


@pytest.mark.parametrize("name,w,layout", CASES, ids=[c[0] for c in CASES])
def test_device_encoder_matches_oracle(dev, w12mod, oracle, name, w, layout):
    od, oblob = oracle.encode(w, layout)
    d, blob_d = w12mod.encode_device(_to_dev(w, dev), layout)
    assert (d.version, d.K, d.N, d.G, d.tiles, d.unit_bytes, d.n_units, d.off_units, d.off_esc, d.n_esc,
            d.total_bytes) == (od.version, od.K, od.N, od.G, od.tiles, od.unit_bytes, od.n_units, od.off_units,
                               od.off_esc, od.n_esc, od.total_bytes)
    got = blob_d.cpu().numpy()
    if not np.array_equal(got, oblob):
        bad = np.nonzero(got != oblob)[0]
        pytest.fail(f"{name}: {bad.size} bytes differ, first at {bad[0]}")
    assert w12mod.validate(d, got) == w12mod.OK


def test_device_encoder_reuse_and_decode(dev, w12mod):
    """Two encodes in a row (the workspace is reused by the binding's fresh
    allocations) and the device decode of the device blob gives W back."""
    import torch
    rng = synth.streams(42, 2)
    for i in range(2):
        w = synth.weights(rng[i], 640, 257)
        d, blob_d = w12mod.encode_device(_to_dev(w, dev), w12mod.LAYOUT_NK)
        out = torch.empty(w.shape, dtype=torch.int16, device=dev)
        w12mod.decode(d, blob_d, out, w12mod.LAYOUT_NK)
        np.testing.assert_array_equal(out.cpu().numpy().view(np.uint16), w)


def test_device_encoder_empty_and_errors(dev, w12mod):
    import torch
    d, blob_d = w12mod.encode_device(torch.empty((0, 256), dtype=torch.int16, device=dev))
    assert d.N == 0 and d.total_bytes == 0 and blob_d.numel() == 0
    with pytest.raises(w12mod.W12Error) as e:
        w12mod.encode_device(torch.zeros((4, 100), dtype=torch.int16, device=dev))
    assert e.value.status == w12mod.ERR_SHAPE
    x = torch.zeros(4 * 128 + 8, dtype=torch.int16, device=dev)
    with pytest.raises(w12mod.W12Error) as e:
        w12mod.encode_device(x[1:1 + 4 * 128].view(4, 128))  # not 16-byte aligned
    assert e.value.status == w12mod.ERR_ALIGN
