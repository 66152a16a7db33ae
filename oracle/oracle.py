"""ctypes wrapper around oracle.c, the float64 CPU oracle (test infrastructure only).

The arithmetic lives in oracle.c; this module only builds it with gcc, loads it and moves
numpy arrays in and out.  See oracle.c for what is computed and which passages of the pages
it follows ("gemm, f32" kernel listing and epilogue; "gemm on tensor cores", section
"What changes"; the matrix-multiplication lab, Part 2, float64 reference).

Nothing here touches a GPU, and nothing in the CUDA library imports this module.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (OpenMP if gcc has it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, f32, vp, ci = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int
            lib.oracle_gemm.argtypes = [i64, i64, i64, f32, vp, vp, f32, vp, vp, vp, ci]
            lib.oracle_gemm.restype = ci
            lib.oracle_gemm_at.argtypes = [i64, i64, i64, f32, vp, vp, f32, vp, vp, vp, i64,
                                           vp, vp, ci]
            lib.oracle_gemm_at.restype = ci
            lib.oracle_gemm_f16out.argtypes = [i64, i64, i64, f32, vp, vp, f32, vp, vp, vp, ci]
            lib.oracle_gemm_f16out.restype = ci
            lib.oracle_f64_to_f16_bits.argtypes = [ctypes.c_double]
            lib.oracle_f64_to_f16_bits.restype = ctypes.c_uint16
            lib.oracle_f32_to_f16.argtypes = [vp, vp, i64]
            lib.oracle_f32_to_f16.restype = None
            lib.oracle_round_f16.argtypes = [vp, vp, i64]
            lib.oracle_round_f16.restype = None
            lib.oracle_f16_bits_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_bits_to_f32.restype = f32
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ci
            lib.oracle_set_num_threads.argtypes = [ci]
            lib.oracle_set_num_threads.restype = None
            _lib = lib
    return _lib


def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def f32_to_f16_bits(x) -> np.ndarray:
    """IEEE binary16 bit patterns of x rounded to nearest, ties to even."""
    x = _f32(x)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_f32_to_f16(_ptr(x), _ptr(out), x.size)
    return out


def f16_bits_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    lib = _load()
    return np.array([lib.oracle_f16_bits_to_f32(int(v)) for v in h.ravel()],
                    dtype=np.float32).reshape(h.shape)


def round_f16(x) -> np.ndarray:
    """x rounded to the nearest f16 (ties to even), returned as exact f32 values."""
    x = _f32(x)
    out = np.empty(x.shape, dtype=np.float32)
    _load().oracle_round_f16(_ptr(x), _ptr(out), x.size)
    return out


def gemm(A, B, C, alpha: float, beta: float, f16_inputs: bool = False,
         want_mag: bool = True):
    """Return (D, mag): D = round_f32(alpha * A @ B + beta * C) summed in float64, and
    mag = sum_k |a_ik| |b_kj| (float64) or None.  f16_inputs rounds A and B to f16 first."""
    A, B = _f32(A), _f32(B)
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: A is {A.shape}, B is {B.shape}")
    Cp = _f32(C) if C is not None else np.zeros((M, N), np.float32)
    if Cp.shape != (M, N):
        raise ValueError(f"C is {Cp.shape}, expected {(M, N)}")
    D = np.empty((M, N), dtype=np.float32)
    mag = np.empty((M, N), dtype=np.float64) if want_mag else None
    rc = _load().oracle_gemm(M, N, K, np.float32(alpha), _ptr(A), _ptr(B), np.float32(beta),
                             _ptr(Cp), _ptr(D), _ptr(mag) if want_mag else None,
                             1 if f16_inputs else 0)
    if rc != 0:
        raise MemoryError("oracle_gemm failed")
    return D, mag


def f64_to_f16_bits(x) -> np.ndarray:
    """float64 values rounded to the nearest f16 (ties to even) in one step, as f16 bit
    patterns (uint16)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    fn = _load().oracle_f64_to_f16_bits
    out = np.fromiter((fn(float(v)) for v in x.reshape(-1)), dtype=np.uint16, count=x.size)
    return out.reshape(x.shape)


def gemm_f16out(A, B, C, alpha: float, beta: float, f16_inputs: bool = False, want_mag: bool = True):
    """Return (D16, mag): D16 = round_f16(alpha * A @ B + beta * C) as f16 bit patterns
    (uint16), summed in float64 with one final rounding; mag as in gemm.  A, B and C are
    given as f32 values (f16 operands held exactly)."""
    A, B = _f32(A), _f32(B)
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: A is {A.shape}, B is {B.shape}")
    Cp = _f32(C) if C is not None else np.zeros((M, N), np.float32)
    if Cp.shape != (M, N):
        raise ValueError(f"C is {Cp.shape}, expected {(M, N)}")
    D = np.empty((M, N), dtype=np.uint16)
    mag = np.empty((M, N), dtype=np.float64) if want_mag else None
    rc = _load().oracle_gemm_f16out(M, N, K, np.float32(alpha), _ptr(A), _ptr(B), np.float32(beta),
                                    _ptr(Cp), _ptr(D), _ptr(mag) if want_mag else None,
                                    1 if f16_inputs else 0)
    if rc != 0:
        raise MemoryError("oracle_gemm_f16out failed")
    return D, mag


def gemm_at(A, B, C, alpha: float, beta: float, rows, cols, f16_inputs: bool = False):
    """The same definition evaluated only at (rows[t], cols[t]).  Returns (values, mag)."""
    A, B = _f32(A), _f32(B)
    M, K = A.shape
    _, N = B.shape
    Cp = _f32(C) if C is not None else np.zeros((1,), np.float32)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    out = np.empty(r.shape, dtype=np.float32)
    mag = np.empty(r.shape, dtype=np.float64)
    rc = _load().oracle_gemm_at(M, N, K, np.float32(alpha), _ptr(A), _ptr(B), np.float32(beta),
                                _ptr(Cp), _ptr(r), _ptr(c), r.size, _ptr(out), _ptr(mag),
                                1 if f16_inputs else 0)
    if rc != 0:
        raise IndexError("oracle_gemm_at: index out of range")
    return out, mag
