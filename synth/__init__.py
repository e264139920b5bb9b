"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle runs.

This module draws random numbers and nothing else: it holds none of the MXFP8
arithmetic (no quantization, no scaling rule, no matmul). Both the CPU oracle
and the CUDA path receive the very same bytes from here.

Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) used as a counter-based stream: draw i of stream
(seed, tag) is mix64(base + (i + 1) * GOLDEN), base = mix64(seed * 2^32 + tag).
Normals come from Box-Muller (Box & Muller 1958) in float64, rounded to float32
and then to bfloat16 with round-to-nearest-even on the bit pattern.

The value recipe follows the decode-projection workloads: entries N(0, 1), each
32-element block along K multiplied by 2**u with u a uniform integer.
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= _M1
        z ^= z >> np.uint64(27)
        z *= _M2
        z ^= z >> np.uint64(31)
    return z


def u64(seed: int, tag: int, n: int) -> np.ndarray:
    """n raw 64-bit draws of stream (seed, tag)."""
    base = _mix64(np.array([(seed << 32) + tag], dtype=np.uint64))[0]
    idx = np.arange(1, n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(base + idx * GOLDEN)


def uniform01(seed: int, tag: int, n: int) -> np.ndarray:
    """Uniform float64 in (0, 1]: the top 53 bits, plus one ulp."""
    return ((u64(seed, tag, n) >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0**-53


def randint(seed: int, tag: int, n: int, lo: int, hi: int) -> np.ndarray:
    """Uniform integers in [lo, hi] (inclusive) as int64."""
    u = uniform01(seed, tag, n)
    k = np.minimum(np.floor(u * (hi - lo + 1)), hi - lo).astype(np.int64)
    return k + lo


def normal(seed: int, tag: int, n: int) -> np.ndarray:
    """n standard normals in float64 (Box-Muller, cosine branch)."""
    u1 = uniform01(seed, tag, n)
    u2 = uniform01(seed, tag + 0x5A5A, n)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> float32 -> bfloat16 bit patterns (uint16), nearest-even on the bits."""
    f = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (f >> np.uint32(16)) & np.uint32(1)
    r = (f + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact value of bfloat16 bit patterns, as float64."""
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def block_scaled_bf16(seed: int, tag: int, rows: int, k: int, umin: int, umax: int) -> np.ndarray:
    """bf16 bit patterns [rows, k]: N(0,1) times 2**u per 32-element block along k,
    u uniform in [umin, umax]. k must be a multiple of 32."""
    assert k % 32 == 0
    z = normal(seed, tag, rows * k).reshape(rows, k // 32, 32)
    u = randint(seed, tag + 1, rows * (k // 32), umin, umax).reshape(rows, k // 32, 1)
    return to_bf16_bits((z * np.exp2(u.astype(np.float64))).reshape(rows, k))


def normal_bf16(seed: int, tag: int, shape) -> np.ndarray:
    """bf16 bit patterns of N(0, 1) draws with the given shape."""
    n = int(np.prod(shape))
    return to_bf16_bits(normal(seed, tag, n)).reshape(shape)


def positions(seed: int, tag: int, t: int, max_pos: int = 65536) -> np.ndarray:
    """t integer token positions uniform in [0, max_pos - 1], int64."""
    return randint(seed, tag, t, 0, max_pos - 1)


def rope_cos_sin_cache(max_pos: int = 65536, rope_dim: int = 64, base: float = 10000.0) -> np.ndarray:
    """The rotary table a model owns and hands to the output projection as an
    input: float32 [max_pos, rope_dim], row p = [cos(p f_0..f_{d/2-1}) | sin(...)]
    with f_i = base**(-2i/rope_dim), evaluated in float64 and rounded once."""
    half = rope_dim // 2
    f = base ** (-2.0 * np.arange(half, dtype=np.float64) / rope_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * f[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


# Tags keep the tensors of one workload on independent streams.
TAG_A, TAG_W, TAG_W2, TAG_W3, TAG_X, TAG_POS, TAG_WOA, TAG_WOB, TAG_NORM = (
    1 << 8, 2 << 8, 3 << 8, 4 << 8, 5 << 8, 6 << 8, 7 << 8, 8 << 8, 9 << 8)


def norm_weight_bf16(seed: int, k: int) -> np.ndarray:
    """bf16 bits of a norm weight vector, uniform in [0.5, 1.5)."""
    return to_bf16_bits(0.5 + uniform01(seed, TAG_NORM, k))
