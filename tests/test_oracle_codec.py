"""Pins of the oracle's W12 codec against facts that do not come from the oracle.

- Round trip: decode(encode(W)) == W for every one of the 65 536 bf16 bit
  patterns (in order and shuffled), in both input orientations.  The pages
  call the format lossless and bit-exact (SpecPilot summary p5 "Reasons"
  bullet 2; p4 "项目介绍" paragraph 2).
- Hand-worked blobs (tests/golden/): the written v1 layout, byte for byte.
- Base rule: closed forms on constructed groups, and a brute-force window
  count (histogram + sliding sum) on random groups: the chosen base attains
  the maximum coverage, is the largest base that does, and the number of
  escapes equals 128 minus that coverage.
"""
import os

import numpy as np
import pytest

from lossless_bit_weight_w12_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _exp(v):
    return (np.asarray(v, dtype=np.uint32) >> 7) & 0xFF


def _all_patterns():
    return np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


@pytest.mark.parametrize("shape", [(65536, 1), (128, 512), (1024, 64)])
@pytest.mark.parametrize("shuffle", [False, True])
@pytest.mark.parametrize("layout", [0, 1])
def test_roundtrip_all_bf16_patterns(oracle, shape, shuffle, layout):
    v = _all_patterns()
    if shuffle:
        v = np.random.default_rng(7).permutation(v)
    K, N = shape
    if layout == oracle.LAYOUT_KN:
        w = v.reshape(K, N)
    else:
        w = v.reshape(N, K)
    d, blob = oracle.encode(w, layout)
    assert d.K == K and d.N == N and d.G == N * (K // 128)
    back = oracle.decode(d, blob, layout)
    assert back.dtype == np.uint16
    np.testing.assert_array_equal(back, w)
    # the other orientation gives the transpose
    other = oracle.decode(d, blob, 1 - layout)
    np.testing.assert_array_equal(other, w.T)


def test_roundtrip_recipe_and_escape_count(oracle):
    rng = synth.streams(0, 1)[0]
    w = synth.weights(rng, 1024, 96)  # [N, K]
    d, blob = oracle.encode(w, oracle.LAYOUT_NK)
    np.testing.assert_array_equal(oracle.decode(d, blob, oracle.LAYOUT_NK), w)
    # escapes: 128 - (max window coverage) per group, counted by brute force
    total = 0
    for n in range(w.shape[0]):
        for kg in range(w.shape[1] // 128):
            e = _exp(w[n, kg * 128:(kg + 1) * 128])
            hist = np.bincount(e, minlength=256)
            cover = np.array([hist[b:b + 15].sum() for b in range(241)])
            total += 128 - cover.max()
    assert d.n_esc == total
    assert total > 0  # the recipe plants zeros and subnormals


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            vals[k] = v
    return vals


def _hexbytes(s):
    return bytes(int(t, 16) for t in s.split()) if s else b""


@pytest.mark.parametrize("name", sorted(f for f in os.listdir(GOLDEN) if f.startswith("example")))
def test_golden_blob(oracle, name):
    """The oracle's blob equals, byte for byte, a layout derived by hand from
    the written format (derivations in the fixture files)."""
    g = _read_golden(name)
    K, N = int(g["K"]), int(g["N"])
    w = np.full((K, N), int(g["weights_rest"], 16), dtype=np.uint16)
    for item in g["weights_at"].split():
        kn, v = item.split(":")
        k, n = (int(t) for t in kn.split(","))
        w[k, n] = int(v, 16)
    d, blob = oracle.encode(w, oracle.LAYOUT_KN)
    raw = blob.tobytes()
    want_desc = [int(t) for t in g["desc"].split()]
    assert [d.tiles, d.unit_bytes, d.n_units, d.off_units, d.off_esc, d.n_esc, d.total_bytes] == want_desc
    assert d.G == N * (K // 128)
    # every plane byte: the listed value, else plane_rest (real columns) or 0 (padding)
    listed = {int(o): int(v, 16) for o, v in (t.split(":") for t in g["bytes"].split())}
    rest = _hexbytes(g["plane_rest"])
    for u in range(d.n_units):
        t = u // (K // 128)
        for plane in range(3):
            for c in range(128):
                real = t * 128 + c < N
                row0 = u * d.unit_bytes + plane * 8192 + 64 * c
                for o in range(row0, row0 + 64):
                    want = listed.get(o, rest[plane] if real else 0)
                    assert raw[o] == want, f"{name}: byte {o} (unit {u}, plane {plane}, column {c})"
    for o in listed:
        assert raw[o] == listed[o]
    for item in g["meta"].split():
        uw, v = item.split(":")
        u, word = (int(x) for x in uw.split(","))
        at = u * d.unit_bytes + 24576 + 4 * word
        assert int.from_bytes(raw[at:at + 4], "little") == int(v, 16), f"{name}: meta {u},{word}"
    for u in range(d.n_units):  # the 12 bytes after the meta words are zero
        at = u * d.unit_bytes + 24576 + 4 * 129
        assert raw[at:at + 12] == bytes(12)
    esc = _hexbytes(g["esc"])
    assert raw[d.off_esc:d.off_esc + len(esc)] == esc
    assert oracle.group_base(w[:128, 0]) == int(g["base"])
    np.testing.assert_array_equal(oracle.decode(d, blob, oracle.LAYOUT_KN), w)


def _group(exps, sign=0, man=0):
    e = np.asarray(exps, dtype=np.uint32)
    return ((sign << 15) | (e << 7) | man).astype(np.uint16)


def test_base_closed_forms(oracle):
    # span <= 14: the window starting at the minimum holds everything
    assert oracle.group_base(_group(np.r_[[100] * 64, [110] * 64])) == 100
    # one value everywhere: b = e, clamped to 240 at the top
    assert oracle.group_base(_group([77] * 128)) == 77
    assert oracle.group_base(_group([0] * 128)) == 0           # all +0
    # the base stops at 240 (so b + 15 fits a byte): a group of Inf/NaN
    # (e = 255) is covered by no window; every window ties at 0 -> b = 240
    assert oracle.group_base(_group([255] * 128)) == 240
    assert oracle.group_base(_group([250] * 128)) == 240       # window [240, 254]
    assert oracle.group_base(_group([254] * 128)) == 240
    # two clusters 20 apart: the larger cluster wins; largest b covering it
    assert oracle.group_base(_group(np.r_[[100] * 100, [120] * 28])) == 100
    assert oracle.group_base(_group(np.r_[[100] * 28, [120] * 100])) == 120
    # a 64/64 tie between the clusters: the larger b
    assert oracle.group_base(_group(np.r_[[100] * 64, [120] * 64])) == 120
    # three clusters: {100 x 50, 110 x 30, 125 x 48}: [100,114] covers 80,
    # [111,125] covers 48, [110,124] covers 30 -> 100
    assert oracle.group_base(_group(np.r_[[100] * 50, [110] * 30, [125] * 48])) == 100


def test_base_bruteforce_random(oracle):
    rng = np.random.default_rng(3)
    for trial in range(300):
        centre = rng.integers(0, 256)
        spread = rng.integers(1, 40)
        e = np.clip(rng.normal(centre, spread, 128).round(), 0, 255).astype(np.uint32)
        vals = _group(e, sign=int(rng.integers(0, 2)), man=int(rng.integers(0, 128)))
        b = oracle.group_base(vals)
        hist = np.bincount(e, minlength=256)
        cover = np.array([hist[x:x + 15].sum() for x in range(241)])
        assert 0 <= b <= 240
        assert cover[b] == cover.max()
        assert b == int(np.flatnonzero(cover == cover.max()).max())


def test_plan_rejects_bad_shapes(oracle):
    w = np.zeros((100, 4), dtype=np.uint16)  # K = 100 is not a multiple of 128
    with pytest.raises(oracle.OracleError) as e:
        oracle.plan(w, oracle.LAYOUT_KN)
    assert e.value.status == oracle.ERR_SHAPE


def test_empty_matrices(oracle):
    for shape in [(0, 5), (128, 0), (0, 0)]:
        w = np.zeros(shape, dtype=np.uint16)
        d, blob = oracle.encode(w, oracle.LAYOUT_KN)
        assert d.G == 0 and d.n_esc == 0
        back = oracle.decode(d, blob)
        assert back.shape == shape


def test_decode_rejects_corrupt_escape_list(oracle):
    w = np.full((128, 1), 0x3F80, dtype=np.uint16)
    w[9, 0] = 0x0000  # one escape
    d, blob = oracle.encode(w)
    bad = blob.copy()
    # point column 0's escape range (meta word 1 of unit 0) past the list
    meta = bad[24576:24576 + 8].view(np.uint32)
    meta[1] = (5 << 8)
    with pytest.raises(oracle.OracleError) as e:
        oracle.decode(d, bad)
    assert e.value.status == oracle.ERR_BLOB
    bad = blob.copy()
    bad[d.off_esc] = 10  # entry now names pos 10, so pos 9 has no entry
    with pytest.raises(oracle.OracleError):
        oracle.decode(d, bad)
