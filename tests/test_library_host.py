"""CPU-side checks of libw12.so: it loads, exports every declared symbol, and
its host encoder and validator agree with the oracle (no device calls)."""
import ctypes
import os
import re

import numpy as np
import pytest

from lossless_bit_weight_w12_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def w12():
    from lossless_bit_weight_w12_gb300 import build_lib, w12 as mod
    build_lib.build()
    mod.lib()
    return mod


def test_exports_every_declared_symbol(w12):
    with open(os.path.join(ROOT, "include", "w12.h")) as f:
        header = f.read()
    declared = set(re.findall(r"\b(w12_[a-z_0-9]+)\s*\(", header))
    assert declared == set(w12.EXPORTS)
    L = ctypes.CDLL(w12.LIB_PATH)
    for name in declared:
        assert hasattr(L, name), name
    assert w12.version() == 2
    assert w12.status_string(w12.ERR_SHAPE).startswith("W12_ERR_SHAPE")


def _cases():
    rng = synth.streams(21, 4)
    yield "recipe_nk", synth.weights(rng[0], 1024, 40), 1
    yield "recipe_kn", np.ascontiguousarray(synth.weights(rng[1], 512, 33).T), 0
    yield "random_bits", synth.random_bits(rng[2], (24, 384)), 1
    allp = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    yield "all_patterns", np.random.default_rng(1).permutation(allp).reshape(128, 512), 1
    yield "all_patterns_ordered", allp.reshape(512, 128), 1


@pytest.mark.parametrize("name,w,layout", list(_cases()), ids=[c[0] for c in _cases()])
def test_encoder_matches_oracle_bytes(w12, oracle, name, w, layout):
    d, blob = w12.encode(w, layout)
    od, oblob = oracle.encode(w, layout)
    assert (d.K, d.N, d.G, d.n_esc, d.total_bytes) == (od.K, od.N, od.G, od.n_esc, od.total_bytes)
    assert (d.tiles, d.unit_bytes, d.n_units, d.off_units, d.off_esc) == \
        (od.tiles, od.unit_bytes, od.n_units, od.off_units, od.off_esc)
    assert blob.tobytes() == oblob.tobytes()
    assert w12.validate(d, blob) == w12.OK
    # the oracle decodes the library's blob back to the input
    np.testing.assert_array_equal(oracle.decode(od, blob, layout), w)


def test_encoder_shape_errors(w12):
    with pytest.raises(w12.W12Error) as e:
        w12.encode_plan(np.zeros((4, 100), np.uint16), w12.LAYOUT_NK)
    assert e.value.status == w12.ERR_SHAPE
    d = w12.encode_plan(np.zeros((0, 128), np.uint16), w12.LAYOUT_NK)
    assert d.G == 0 and d.N == 0


def test_validate_catches_corruption(w12):
    rng = synth.streams(22, 1)[0]
    w = synth.weights(rng, 512, 16)
    d, blob = w12.encode(w, w12.LAYOUT_NK)
    assert d.n_esc > 0
    meta_at = 3 * 8192  # meta words of a unit block
    last = (d.n_units - 1) * d.unit_bytes + meta_at
    bad = blob.copy()
    bad[meta_at] = 250  # base of column 0 of unit 0 above 240
    assert w12.validate(d, bad) == w12.ERR_BLOB
    bad = blob.copy()
    meta = bad[last:last + 4 * 129].view(np.uint32)
    meta[128] += 1 << 8  # the last unit's end no longer n_esc
    assert w12.validate(d, bad) == w12.ERR_BLOB
    bad = blob.copy()
    meta = bad[meta_at:meta_at + 4 * 129].view(np.uint32)
    meta[20] = 0  # a padding column (N = 16) with a base or escapes
    meta[20] |= 3
    assert w12.validate(d, bad) == w12.ERR_BLOB
    bad = blob.copy()
    bad[8192 * 2 + 64 * 40 + 3] = 0x10  # plane bytes in a padding column
    assert w12.validate(d, bad) == w12.ERR_BLOB
    bad = blob.copy()
    esc = bad[d.off_esc:d.off_esc + 2 * d.n_esc].view(np.uint16)
    esc[0] ^= 1  # an escape moved to another position
    assert w12.validate(d, bad) == w12.ERR_BLOB
    bad = blob.copy()
    e0 = 2 * 8192  # E plane block of unit 0, column 0's row
    i = next(j for j in range(e0, e0 + 64) if (blob[j] & 0x0F) != 0x0F)
    bad[i] |= 0x0F  # a code-15 nibble with no escape entry
    assert w12.validate(d, bad) == w12.ERR_BLOB
    assert w12.validate(d, blob) == w12.OK
