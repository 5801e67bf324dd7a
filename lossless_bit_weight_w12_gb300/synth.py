"""Seeded synthetic workloads shared by the tests, the oracle checks and the bench.

This module only draws numbers; it holds none of the W12 arithmetic (no
encoding, no decoding, no products).  Every tensor gets its own random stream:
``numpy.random.SeedSequence(seed).spawn(n)[i]`` for the i-th tensor in listed
order, so tensors can be drawn independently and in any order.

Weight recipe (a dense decoder layer's linears in bf16):
  1. fp32 draws from N(0, 0.02), rounded to bf16 round-to-nearest-even;
  2. outliers: Binomial(size, 1e-3) positions (uniform, with replacement)
     are multiplied by 64 (exact in bf16: the exponent grows by 6);
  3. specials: Binomial(size, 1e-4) positions are overwritten, half by +-0,
     half by a subnormal with mantissa uniform on 1..127, each with a random
     sign.
Activations: fp32 N(0, 1) rounded to bf16 the same way.

Weights are returned in the [N, K] (out x in) orientation of a linear
layer's weight, as bf16 bit patterns in uint16.
"""
from __future__ import annotations

import numpy as np

# One dense 27B-class decoder layer, hidden 5120: (name, K = in, N = out).
LAYER_SHAPES = (
    ("q", 5120, 6144),
    ("k", 5120, 1024),
    ("v", 5120, 1024),
    ("o", 6144, 5120),
    ("gate_up", 5120, 2 * 17408),
    ("down", 17408, 5120),
)
LM_HEAD_SHAPE = ("lm_head", 5120, 151936)
N_LAYERS_STACK = 64


def layer_shapes():
    return list(LAYER_SHAPES)


def weight_bytes_w12(K: int, N: int) -> float:
    """Algorithmic W12 bytes of a K x N weight: 12 bits per weight."""
    return 1.5 * K * N


def streams(seed: int, n: int):
    """n independent generators for seed, one per tensor in listed order."""
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]


def bf16_rne(f: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns bit patterns."""
    b = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    nan = (b & 0x7FFFFFFF) > 0x7F800000
    r = ((b + np.uint32(0x7FFF) + ((b >> 16) & np.uint32(1))) >> 16).astype(np.uint16)
    if nan.any():
        r[nan] = ((b[nan] >> 16) | 0x0040).astype(np.uint16)
    return r


def bf16_to_f32(u: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def weights(rng: np.random.Generator, K: int, N: int, std: float = 0.02,
            p_outlier: float = 1e-3, outlier_scale: float = 64.0,
            p_special: float = 1e-4) -> np.ndarray:
    """[N, K] bf16 weight following the recipe in the module docstring."""
    size = K * N
    # The normal draws are taken in chunks (the same sequence as one draw of
    # `size`) and rounded while they are in cache.
    w = np.empty(size, dtype=np.uint16)
    chunk = 1 << 20
    for c0 in range(0, size, chunk):
        f = rng.standard_normal(min(chunk, size - c0), dtype=np.float32)
        f *= np.float32(std)
        w[c0:c0 + f.size] = bf16_rne(f)
    if size:
        n_out = int(rng.binomial(size, p_outlier))
        at = rng.integers(0, size, n_out)
        w[at] = bf16_rne(bf16_to_f32(w[at]) * np.float32(outlier_scale))
        n_sp = int(rng.binomial(size, p_special))
        at = rng.integers(0, size, n_sp)
        kind = rng.integers(0, 2, n_sp)
        sign = rng.integers(0, 2, n_sp).astype(np.uint16) << 15
        mant = rng.integers(1, 128, n_sp).astype(np.uint16)
        w[at] = np.where(kind == 0, sign, sign | mant).astype(np.uint16)
    return w.reshape(N, K)


def activations(rng: np.random.Generator, M: int, K: int) -> np.ndarray:
    """[M, K] bf16 activations, N(0, 1)."""
    return bf16_rne(rng.standard_normal(M * K, dtype=np.float32)).reshape(M, K)


def random_bits(rng: np.random.Generator, shape) -> np.ndarray:
    """Uniformly random 16-bit patterns (every bf16 class: NaN, Inf, subnormal)."""
    return rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)


def logits(rng: np.random.Generator, rows: int, V: int, dtype=np.float32) -> np.ndarray:
    """[rows, V] logits ~ N(0, 4) in float32 (or bf16 bits when dtype is uint16)."""
    f = rng.standard_normal(rows * V, dtype=np.float32) * np.float32(2.0)
    f = f.reshape(rows, V)
    return bf16_rne(f) if dtype == np.uint16 else f


def draft_tokens(rng: np.random.Generator, target: np.ndarray, R: int, T: int, V: int,
                 p_match: float = 0.7) -> np.ndarray:
    """[R, T-1] drafts: position i agrees with target[r, i] with probability p_match
    while every earlier one agreed (a geometric prefix, capped at T-1); the
    first disagreeing token is uniform on [0, V) redrawn until it differs;
    later tokens are uniform.  ``target`` is [R, T] (the target's greedy
    token per position), supplied by the caller."""
    target = np.asarray(target).reshape(R, T)
    d = rng.integers(0, V, size=(R, max(T - 1, 0))).astype(np.int32)
    for r in range(R):
        for i in range(T - 1):
            if rng.random() < p_match:
                d[r, i] = target[r, i]
                continue
            t = int(rng.integers(0, V))
            while t == int(target[r, i]) and V > 1:
                t = int(rng.integers(0, V))
            d[r, i] = t
            break
    return d
