"""Seeded synthetic inputs shared by the tests, the oracle checks and the benchmark.

This module draws numbers and nothing else: it holds none of the GEMM's arithmetic.  Every
value is a pure function of (seed, tensor id, element index), so any element of any
matrix can be regenerated on its own and both sides of a parity check see the same bits.

Generator: the splitmix64 output function (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; constants as in Vigna's public-domain
reference code), used as a counter-based hash:

    mix(z)      = z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
                  z *= 0x94D049BB133111EB; z ^= z >> 31
    key(s, t)   = mix((256 * s + t) * G)          G = 0x9E3779B97F4A7C15
    h(s, t, i)  = mix(key(s, t) + (i + 1) * G)     all arithmetic mod 2^64

Distributions (row-major linear index i):

    "uniform"   x = (h >> 40) * 2^-23 - 1     uniform on [-1, 1), a 2^-23 grid exact in f32
    "unit"      x = (h >> 40) * 2^-24         uniform on [0, 1), exact in f32
    "int3"      x = ((h >> 32) mod 7) - 3     integers in {-3, ..., 3}
    "f16grid"   x = (h >> 53) * 2^-10 - 1     uniform on [-1, 1), a 2^-10 grid exact in f16
                                              (inputs for the half-precision entry points)

The pages' workloads are i.i.d. dense random matrices (uniform [0,1) in the lab's ladder,
uniform [-0.5, 0.5) in its precision study, normal in its cuBLAS sweeps); the workloads
here use "uniform" on [-1, 1) with seed 0 and tensor ids A=0, B=1, C=2.
"""
from __future__ import annotations

import numpy as np

TENSOR_A, TENSOR_B, TENSOR_C = 0, 1, 2
DISTRIBUTIONS = ("uniform", "unit", "int3", "f16grid")

_G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _M1
    z = z ^ (z >> np.uint64(27))
    z = z * _M2
    return z ^ (z >> np.uint64(31))


def _mix_scalar(z: int) -> int:
    mask = (1 << 64) - 1
    z &= mask
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & mask
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & mask
    return z ^ (z >> 31)


def key(seed: int, tensor: int) -> int:
    return _mix_scalar(((256 * int(seed) + int(tensor)) * 0x9E3779B97F4A7C15) & ((1 << 64) - 1))


def hashes(seed: int, tensor: int, start: int, count: int) -> np.ndarray:
    """h(seed, tensor, i) for i in [start, start + count), as uint64."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
        return _mix(np.uint64(key(seed, tensor)) + i * _G)


def _values(h: np.ndarray, dist: str) -> np.ndarray:
    if dist == "uniform":
        return ((h >> np.uint64(40)).astype(np.float64) * 2.0 ** -23 - 1.0).astype(np.float32)
    if dist == "unit":
        return ((h >> np.uint64(40)).astype(np.float64) * 2.0 ** -24).astype(np.float32)
    if dist == "int3":
        return (((h >> np.uint64(32)) % np.uint64(7)).astype(np.int64) - 3).astype(np.float32)
    if dist == "f16grid":
        return ((h >> np.uint64(53)).astype(np.float64) * 2.0 ** -10 - 1.0).astype(np.float32)
    raise ValueError(f"unknown distribution {dist!r}; expected one of {DISTRIBUTIONS}")


def fill(out: np.ndarray, seed: int, tensor: int, dist: str = "uniform") -> np.ndarray:
    """Fill the contiguous float32 array ``out`` in place (row-major linear index)."""
    if out.dtype != np.float32 or not out.flags["C_CONTIGUOUS"]:
        raise ValueError("out must be a C-contiguous float32 array")
    flat = out.reshape(-1)
    n = flat.size
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        flat[s:s + c] = _values(hashes(seed, tensor, s, c), dist)
    return out


def matrix(rows: int, cols: int, seed: int = 0, tensor: int = TENSOR_A,
           dist: str = "uniform") -> np.ndarray:
    """A new rows x cols float32 matrix from the generator."""
    return fill(np.empty((rows, cols), dtype=np.float32), seed, tensor, dist)


def problem(M: int, N: int, K: int, seed: int = 0, dist: str = "uniform"):
    """(A, B, C) for one GEMM: A is M x K, B is K x N, C is M x N."""
    return (matrix(M, K, seed, TENSOR_A, dist), matrix(K, N, seed, TENSOR_B, dist),
            matrix(M, N, seed, TENSOR_C, dist))
