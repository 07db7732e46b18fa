"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the GEMM or of the quantizers: it only
draws normal variates and rounds them to bf16.  Both the CUDA path and the
CPU oracle receive the arrays it returns.

Generator (stated so that any reimplementation reproduces it bit for bit):

* SplitMix64 as a counter-based generator: output i of stream ``seed`` is the
  SplitMix64 finaliser applied to ``seed * G + (i + 1) * G`` (mod 2^64) with
  G = 0x9E3779B97F4A7C15.
* 53-bit uniforms u = (z >> 11) * 2^-53.
* Box-Muller on the pair (u[2j], u[2j+1]):
  r = sqrt(-2 ln(1 - u[2j])), n[2j] = r cos(2 pi u[2j+1]),
  n[2j+1] = r sin(2 pi u[2j+1]), all in fp64.
* x = mean + std * n in fp64, rounded to fp32 (nearest-even) and then to
  bf16 (nearest-even).

The value distributions are the ones the workloads name: activations and
residuals N(0, 1), weights N(0, 1) or N(0, 0.02).  Seeds: A = 0, W = 1,
residual = 2 unless a test says otherwise.
"""
from __future__ import annotations

import numpy as np

_G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 24


def _splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z = np.uint64(seed) * _G + i * _G
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def normal_f64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """n standard normals (fp64) of stream ``seed`` starting at variate ``start`` (even)."""
    assert start % 2 == 0
    m = n + (n & 1)
    z = _splitmix64(seed, start, m)
    u = (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log1p(-u1))
    th = 2.0 * np.pi * u2
    out = np.empty(m, np.float64)
    out[0::2] = r * np.cos(th)
    out[1::2] = r * np.sin(th)
    return out[:n]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest-even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(shape, seed: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(mean, std^2) variates, row-major ``shape``."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    out = np.empty(n, np.uint16)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        x = mean + std * normal_f64(seed, c, start=s)
        out[s:s + c] = f32_to_bf16_bits(x.astype(np.float32))
    return out.reshape(shape)


def random_codes(shape, seed: int, exclude=()) -> np.ndarray:
    """Uniform random bytes (for code-level tests), skipping the values in ``exclude``."""
    n = int(np.prod(shape))
    z = _splitmix64(seed, 0, 2 * n + 64)
    b = (z & np.uint64(0xFF)).astype(np.uint8)
    if exclude:
        b = b[~np.isin(b, np.asarray(exclude, np.uint8))]
    assert b.size >= n
    return b[:n].reshape(shape)
