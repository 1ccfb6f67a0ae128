"""Seeded synthetic inputs for the routed-expert MoE layer (host side, numpy).

This module holds the input generators only: random codes, scales, weights,
activations and router biases.  It holds none of the layer's arithmetic.
Both the GPU path and the oracle take their inputs from here, and the device
generator in ``csrc/synth_fill.cu`` implements the same counter-based
definition for the multi-gigabyte expert arenas, so that any element can be
regenerated on the host for a sampled check.

The generator (stated once, implemented on both sides):

* ``mix64`` is the SplitMix64 output function (Steele, Lea, Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014):
  ``z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
  z *= 0x94D049BB133111EB; z ^= z >> 31`` (all mod 2^64).
* A stream is named by ``key = stream_key(seed, tag, layer, expert)`` and its
  i-th 64-bit word is ``u64(key, i) = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)``.
* A code of ``bits`` bits is the top ``bits`` bits of ``u64(key, i)``.
* A standard normal is approximated by the Irwin-Hall sum of the eight 16-bit
  halves of ``u64(key, 2i)`` and ``u64(key, 2i+1)``:
  ``z = f32(S - 262140) * f32(1 / (65535 * sqrt(2/3)))`` (one fp32 multiply,
  round-to-nearest-even; the integer difference is exact in fp32).  Its
  support is +-4.9; mean 0, variance 1.
* ``N(0, sigma)`` is ``f32(z * f32(sigma))``; bf16 and fp16 values are the
  round-to-nearest-even of that fp32 number.
"""
from __future__ import annotations

import math

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
M1 = np.uint64(0xBF58476D1CE4E5B9)
M2 = np.uint64(0x94D049BB133111EB)
IH_MEAN = 4 * 65535  # mean of the sum of eight 16-bit uniforms
IH_SCALE = np.float32(1.0 / (65535.0 * math.sqrt(2.0 / 3.0)))

# stream tags
TAG_GU_CODES = 1
TAG_GU_SCALES = 2
TAG_D_CODES = 3
TAG_D_SCALES = 4
TAG_ROUTER = 5
TAG_SHARED_G = 6
TAG_SHARED_U = 7
TAG_SHARED_D = 8
TAG_X = 9
TAG_RANK = 10
TAG_CTX = 11

# Router-bias strength for Zipf popularity: b_e = -kappa * s * ln(rank_e + 1).
# Found by bisection so that, for H=2048, E=512, k=10, router weights
# N(0, 0.02) and activations N(0, 1) from this generator, the log-log slope of
# pick count against rank (ranks picked by fewer than half of 4,096 tokens) is
# -s.  tests/golden/calibrate_zipf.py reproduces these values.
ZIPF_KAPPA = {1.1: 0.3837, 1.4: 0.3630}

_MASK64 = (1 << 64) - 1


def mix64(z):
    """SplitMix64 output function on a numpy uint64 array (wrapping)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = z ^ (z >> np.uint64(30))
        z = z * M1
        z = z ^ (z >> np.uint64(27))
        z = z * M2
        z = z ^ (z >> np.uint64(31))
    return z


def _mix64_int(z: int) -> int:
    z &= _MASK64
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & _MASK64
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tag: int, layer: int = 0, expert: int = 0) -> int:
    """64-bit key of one stream: mix64(mix64(mix64(seed + G) ^ tag) ^ (layer << 32 | expert))."""
    k = _mix64_int((seed + 0x9E3779B97F4A7C15) & _MASK64)
    k = _mix64_int(k ^ (tag & _MASK64))
    return _mix64_int(k ^ (((layer & 0xFFFFFFFF) << 32) | (expert & 0xFFFFFFFF)))


def u64(key: int, idx) -> np.ndarray:
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(np.uint64(key) + (idx + np.uint64(1)) * GOLDEN)


def codes(key: int, n: int, bits: int, start: int = 0) -> np.ndarray:
    """n uniform codes in [0, 2^bits), uint8."""
    w = u64(key, np.arange(start, start + n, dtype=np.uint64))
    return (w >> np.uint64(64 - bits)).astype(np.uint8)


def normal(key: int, n: int, start: int = 0) -> np.ndarray:
    """n approximately standard-normal fp32 values (Irwin-Hall of eight 16-bit uniforms)."""
    i = np.arange(start, start + n, dtype=np.uint64)
    a = u64(key, 2 * i)
    b = u64(key, 2 * i + np.uint64(1))
    s = np.zeros(n, np.int64)
    for w in (a, b):
        for j in range(4):
            s += ((w >> np.uint64(16 * j)) & np.uint64(0xFFFF)).astype(np.int64)
    return (s - IH_MEAN).astype(np.float32) * IH_SCALE


def normal_sigma(key: int, n: int, sigma: float, start: int = 0) -> np.ndarray:
    return normal(key, n, start) * np.float32(sigma)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bit pattern (finite inputs)."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_fp16_bits(a: np.ndarray) -> np.ndarray:
    return np.asarray(a, np.float32).astype(np.float16).view(np.uint16)


# ---------------------------------------------------------------------------
# Tensors of one layer
# ---------------------------------------------------------------------------

def expert_codes(seed, layer, expert, bits, H, I):
    """Logical codes of one expert: gate [I][H], up [I][H], down [H][I] (uint8)."""
    gu = codes(stream_key(seed, TAG_GU_CODES, layer, expert), 2 * I * H, bits).reshape(2, I, H)
    d = codes(stream_key(seed, TAG_D_CODES, layer, expert), H * I, bits).reshape(H, I)
    return gu[0], gu[1], d


def expert_scales(seed, layer, expert, H, I, sigma=0.02):
    """fp16 bit patterns of |N(0, sigma)| scales: gate/up [2][I][H/32], down [H][I/32]."""
    gu = np.abs(normal_sigma(stream_key(seed, TAG_GU_SCALES, layer, expert), 2 * I * (H // 32), sigma))
    d = np.abs(normal_sigma(stream_key(seed, TAG_D_SCALES, layer, expert), H * (I // 32), sigma))
    return (f32_to_fp16_bits(gu).reshape(2, I, H // 32), f32_to_fp16_bits(d).reshape(H, I // 32))


def router_weights(seed, layer, E, H, sigma=0.02):
    return normal_sigma(stream_key(seed, TAG_ROUTER, layer), E * H, sigma).reshape(E, H)


def shared_weights(seed, layer, H, Is, sigma=0.02):
    """bf16 bit patterns: wg [Is][H], wu [Is][H], wd [H][Is]."""
    g = f32_to_bf16_bits(normal_sigma(stream_key(seed, TAG_SHARED_G, layer), Is * H, sigma)).reshape(Is, H)
    u = f32_to_bf16_bits(normal_sigma(stream_key(seed, TAG_SHARED_U, layer), Is * H, sigma)).reshape(Is, H)
    d = f32_to_bf16_bits(normal_sigma(stream_key(seed, TAG_SHARED_D, layer), H * Is, sigma)).reshape(H, Is)
    return g, u, d


def activations(seed, T, H, step=0):
    """x ~ N(0, 1) as bf16 bit patterns [T][H]."""
    return f32_to_bf16_bits(normal(stream_key(seed, TAG_X, step), T * H)).reshape(T, H)


def verify_window(seed, T, H, step=0, noise=0.3):
    """T tokens sharing a context c ~ N(0,1) plus N(0, noise) each, bf16 bits [T][H]."""
    c = normal(stream_key(seed, TAG_CTX, step), H)
    n = normal_sigma(stream_key(seed, TAG_X, step), T * H, noise).reshape(T, H)
    return f32_to_bf16_bits(c[None, :] + n)


def zipf_rank(seed, layer, E):
    """A seeded permutation: rank_e of each expert (0 = most popular)."""
    order = np.argsort(u64(stream_key(seed, TAG_RANK, layer), np.arange(E, dtype=np.uint64)), kind="stable")
    rank = np.empty(E, np.int64)
    rank[order] = np.arange(E)
    return rank


def zipf_bias(seed, layer, E, s, kappa=None):
    """fp32 router bias b_e = -kappa * s * ln(rank_e + 1); zero when s == 0 (uniform routing)."""
    if not s:
        return np.zeros(E, np.float32)
    if kappa is None:
        kappa = ZIPF_KAPPA[s]
    rank = zipf_rank(seed, layer, E)
    return (-kappa * s * np.log(rank + 1.0)).astype(np.float32)
