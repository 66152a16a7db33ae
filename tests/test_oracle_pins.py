"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks the oracle against something independent of it: numpy's binary16
conversion and float64 matmul (library routines), exact integer arithmetic, exact rational
arithmetic (fractions.Fraction), closed forms (identity, alpha = 0, beta = 0, K = 0) and the
error levels the matrix-multiplication lab prints for f16 inputs with f32 accumulation.
A plausible mistake anywhere in the oracle (a dropped term, a wrong sign or index, a
transposed operand, truncation instead of rounding) fails at least one of them.
"""
import os
import random
from fractions import Fraction

import numpy as np
import pytest

from dense_gemm_04_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _bits_f32(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


def _np_f16_bits(x):
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def _same_f16(a, b):
    """Bitwise equality, except that any two NaNs of the same sign count as equal."""
    a = np.asarray(a, dtype=np.uint16)
    b = np.asarray(b, dtype=np.uint16)
    nan_a = ((a & 0x7C00) == 0x7C00) & ((a & 0x03FF) != 0)
    nan_b = ((b & 0x7C00) == 0x7C00) & ((b & 0x03FF) != 0)
    return np.where(nan_a | nan_b, nan_a & nan_b & ((a & 0x8000) == (b & 0x8000)), a == b)


# ----------------------------------------------------------------------------------------
# f32 -> f16 rounding
# ----------------------------------------------------------------------------------------

def test_f16_rounding_golden_cases(oracle_mod):
    rows = _read_table("f16_rounding_cases.txt")
    x = np.array([int(r[0], 16) for r in rows], dtype=np.uint32).view(np.float32)
    want = np.array([int(r[1], 16) for r in rows], dtype=np.uint16)
    got = oracle_mod.f32_to_f16_bits(x)
    bad = [(rows[i][0], hex(got[i]), rows[i][1]) for i in range(len(rows)) if got[i] != want[i]]
    assert not bad, bad


def test_f16_rounding_matches_numpy_every_high_pattern(oracle_mod):
    """Every combination of sign, exponent and the top 10 fraction bits (2^19 patterns),
    each with low 13 bits at the rounding boundaries and at random values."""
    hi = np.arange(1 << 19, dtype=np.uint32) << np.uint32(13)
    rng = np.random.default_rng(1)
    lows = [0x0000, 0x0001, 0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x0800, 0x17FF]
    lows += [int(v) for v in rng.integers(0, 1 << 13, size=8)]
    for low in lows:
        x = (hi | np.uint32(low)).view(np.float32)
        assert _same_f16(oracle_mod.f32_to_f16_bits(x), _np_f16_bits(x)).all(), hex(low)


def test_f16_rounding_matches_numpy_random_and_subnormal(oracle_mod):
    rng = np.random.default_rng(2)
    x = rng.integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32).view(np.float32)
    assert _same_f16(oracle_mod.f32_to_f16_bits(x), _np_f16_bits(x)).all()
    # every f32 exponent whose values land in or next to the f16 subnormal range
    exps = rng.integers(98, 114, size=1 << 22).astype(np.uint32)
    frac = rng.integers(0, 1 << 23, size=1 << 22).astype(np.uint32)
    sign = rng.integers(0, 2, size=1 << 22).astype(np.uint32) << np.uint32(31)
    x = (sign | (exps << np.uint32(23)) | frac).view(np.float32)
    assert _same_f16(oracle_mod.f32_to_f16_bits(x), _np_f16_bits(x)).all()


def test_f16_decode_matches_numpy_all_patterns(oracle_mod):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    want = h.view(np.float16).astype(np.float32)
    got = oracle_mod.f16_bits_to_f32(h)
    both_nan = np.isnan(want) & np.isnan(got)
    assert (both_nan | (_bits_f32(got) == _bits_f32(want))).all()


def test_round_f16_is_nearest(oracle_mod):
    """Brute force on a sample: no other f16 value is strictly closer than the result."""
    x = synth.matrix(64, 64, seed=5, dist="uniform") * np.float32(3.0)
    r = oracle_mod.round_f16(x).astype(np.float64).ravel()
    finite16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    finite16 = np.unique(finite16[np.isfinite(finite16)].astype(np.float64))
    xs = x.astype(np.float64).ravel()
    idx = np.clip(np.searchsorted(finite16, xs), 1, finite16.size - 1)
    best = np.minimum(np.abs(finite16[idx] - xs), np.abs(finite16[idx - 1] - xs))
    assert (np.abs(r - xs) <= best).all()


# ----------------------------------------------------------------------------------------
# GEMM: closed forms
# ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("f16", [False, True])
def test_identity(oracle_mod, f16):
    M = K = 37
    N = 23
    A = np.eye(M, K, dtype=np.float32)
    B = synth.matrix(K, N, seed=3, tensor=1, dist="int3")
    C = synth.matrix(M, N, seed=3, tensor=2, dist="int3")
    D, mag = oracle_mod.gemm(A, B, C, 1.5, 0.5, f16_inputs=f16)
    want = (1.5 * B.astype(np.float64) + 0.5 * C.astype(np.float64)).astype(np.float32)
    assert np.array_equal(_bits_f32(D), _bits_f32(want))
    assert np.array_equal(mag, np.abs(B).astype(np.float64))


@pytest.mark.parametrize("f16", [False, True])
def test_alpha_zero_reads_neither_a_nor_b(oracle_mod, f16):
    M, N, K = 9, 11, 13
    A = np.full((M, K), np.nan, dtype=np.float32)
    B = np.full((K, N), np.nan, dtype=np.float32)
    C = synth.matrix(M, N, seed=4, tensor=2)
    D, _ = oracle_mod.gemm(A, B, C, 0.0, 0.75, f16_inputs=f16)
    want = (0.75 * C.astype(np.float64)).astype(np.float32)
    assert np.array_equal(_bits_f32(D), _bits_f32(want))


@pytest.mark.parametrize("f16", [False, True])
def test_beta_zero_does_not_read_c(oracle_mod, f16):
    M, N, K = 17, 19, 23
    A = synth.matrix(M, K, seed=6, tensor=0, dist="int3")
    B = synth.matrix(K, N, seed=6, tensor=1, dist="int3")
    C = np.full((M, N), np.nan, dtype=np.float32)
    D, _ = oracle_mod.gemm(A, B, C, 2.0, 0.0, f16_inputs=f16)
    want = (2 * (A.astype(np.int64) @ B.astype(np.int64))).astype(np.float32)
    assert not np.isnan(D).any()
    assert np.array_equal(D, want)


def test_k_zero_scales_c(oracle_mod):
    A = np.zeros((5, 0), np.float32)
    B = np.zeros((0, 7), np.float32)
    C = synth.matrix(5, 7, seed=8, tensor=2)
    D, _ = oracle_mod.gemm(A, B, C, 1.5, -2.0)
    assert np.array_equal(D, (-2.0 * C.astype(np.float64)).astype(np.float32))


# ----------------------------------------------------------------------------------------
# GEMM: exact integer arithmetic (numpy int64 matmul is the independent reference)
# ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 7), (65, 33, 129), (128, 96, 300),
                                   (40, 257, 64), (257, 1, 1000), (1, 300, 517)])
@pytest.mark.parametrize("ab", [(1.5, 0.5), (2.0, -1.0), (1.0, 0.0)])
@pytest.mark.parametrize("f16", [False, True])
def test_integer_inputs_exact(oracle_mod, shape, ab, f16):
    M, N, K = shape
    alpha, beta = ab
    A = synth.matrix(M, K, seed=11, tensor=0, dist="int3")
    B = synth.matrix(K, N, seed=11, tensor=1, dist="int3")
    C = synth.matrix(M, N, seed=11, tensor=2, dist="int3")
    S = A.astype(np.int64) @ B.astype(np.int64)
    want = (alpha * S.astype(np.float64) + beta * C.astype(np.float64)).astype(np.float32)
    D, mag = oracle_mod.gemm(A, B, C, alpha, beta, f16_inputs=f16)
    assert np.array_equal(_bits_f32(D), _bits_f32(want))
    assert np.array_equal(mag, (np.abs(A).astype(np.int64) @ np.abs(B).astype(np.int64)).astype(np.float64))


# ----------------------------------------------------------------------------------------
# GEMM: exact rational arithmetic on tiny shapes
# ----------------------------------------------------------------------------------------

def _f32_ulp(v: float) -> float:
    v = abs(np.float32(v))
    return float(np.spacing(v)) if v > 0 else float(np.spacing(np.float32(0)))


@pytest.mark.parametrize("f16", [False, True])
def test_brute_force_tiny_shapes_exact_rationals(oracle_mod, f16):
    rnd = random.Random(7)
    for trial in range(60):
        M, N, K = rnd.randint(1, 4), rnd.randint(1, 4), rnd.randint(1, 4)
        A = synth.matrix(M, K, seed=100 + trial, tensor=0) * np.float32(rnd.choice([1, 3, 1e-3]))
        B = synth.matrix(K, N, seed=100 + trial, tensor=1) * np.float32(rnd.choice([1, 7, 1e3]))
        C = synth.matrix(M, N, seed=100 + trial, tensor=2)
        alpha = float(np.float32(rnd.uniform(-2, 2)))
        beta = float(np.float32(rnd.choice([0.0, rnd.uniform(-2, 2)])))
        Ain = A.astype(np.float16).astype(np.float32) if f16 else A
        Bin = B.astype(np.float16).astype(np.float32) if f16 else B
        D, mag = oracle_mod.gemm(A, B, C, alpha, beta, f16_inputs=f16)
        for i in range(M):
            for j in range(N):
                s = sum(Fraction(float(Ain[i, k])) * Fraction(float(Bin[k, j])) for k in range(K))
                exact = Fraction(alpha) * s + Fraction(beta) * Fraction(float(C[i, j]))
                m = sum(abs(Fraction(float(Ain[i, k])) * Fraction(float(Bin[k, j]))) for k in range(K))
                # one f32 rounding (half an ulp) plus float64 rounding of the sum and epilogue
                slack = 0.5 * _f32_ulp(float(exact)) + 8 * 2.0 ** -53 * (
                    abs(alpha) * float(m) + abs(beta) * abs(float(C[i, j])))
                assert abs(float(D[i, j]) - float(exact)) <= slack, (trial, i, j)
                assert abs(mag[i, j] - float(m)) <= 4 * K * 2.0 ** -53 * float(m)


# ----------------------------------------------------------------------------------------
# GEMM: float64 library matmul on non-square, non-symmetric inputs (catches transposes)
# ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(31, 47, 53), (128, 64, 200), (5, 300, 17), (300, 3, 517), (1, 130, 999)])
def test_matches_numpy_float64(oracle_mod, shape):
    M, N, K = shape
    A, B, C = synth.problem(M, N, K, seed=21)
    alpha, beta = 2.0, -1.0
    ref = alpha * (A.astype(np.float64) @ B.astype(np.float64)) + beta * C.astype(np.float64)
    D, mag = oracle_mod.gemm(A, B, C, alpha, beta)
    # D and ref differ only by float64 summation order and one f32 rounding of the result
    slack = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64) + \
        8 * K * 2.0 ** -53 * (abs(alpha) * mag + abs(beta) * np.abs(C))
    assert (np.abs(D.astype(np.float64) - ref) <= slack).all()
    assert np.allclose(mag, np.abs(A).astype(np.float64) @ np.abs(B).astype(np.float64),
                       rtol=1e-13, atol=0)
    # the f16 variant is the same product of the f16-rounded operands (numpy rounding)
    A16 = A.astype(np.float16).astype(np.float64)
    B16 = B.astype(np.float16).astype(np.float64)
    ref16 = alpha * (A16 @ B16) + beta * C.astype(np.float64)
    D16, mag16 = oracle_mod.gemm(A, B, C, alpha, beta, f16_inputs=True)
    slack16 = np.spacing(np.abs(ref16).astype(np.float32)).astype(np.float64) + \
        8 * K * 2.0 ** -53 * (abs(alpha) * mag16 + abs(beta) * np.abs(C))
    assert (np.abs(D16.astype(np.float64) - ref16) <= slack16).all()


@pytest.mark.parametrize("f16", [False, True])
def test_gemm_at_equals_full_gemm(oracle_mod, f16):
    M, N, K = 70, 90, 110
    A, B, C = synth.problem(M, N, K, seed=31)
    D, mag = oracle_mod.gemm(A, B, C, 1.5, 0.5, f16_inputs=f16)
    rng = np.random.default_rng(0)
    rows = rng.integers(0, M, 500)
    cols = rng.integers(0, N, 500)
    v, m = oracle_mod.gemm_at(A, B, C, 1.5, 0.5, rows, cols, f16_inputs=f16)
    assert np.array_equal(_bits_f32(v), _bits_f32(D[rows, cols]))
    assert np.array_equal(m, mag[rows, cols])


def test_gemm_at_rejects_bad_index(oracle_mod):
    A, B, C = synth.problem(4, 4, 4)
    with pytest.raises(IndexError):
        oracle_mod.gemm_at(A, B, C, 1.0, 0.0, [4], [0])


# ----------------------------------------------------------------------------------------
# The lab's printed error levels for f16 inputs with f32 accumulation
# ----------------------------------------------------------------------------------------

def _errors(out, ref):
    diff = out.astype(np.float64) - ref
    return float(np.abs(diff).max() / np.abs(ref).max()), float(np.linalg.norm(diff) / np.linalg.norm(ref))


def test_f16_variant_error_level_matches_lab(oracle_mod):
    """n = 1024, uniform [0, 1): the lab prints max 5.7e-5 and Frobenius 1.5e-5 for f16
    inputs summed in f32, against float64 of the unrounded inputs.  Rounding to nearest
    reproduces that level; truncating the inputs instead gives a biased error many times
    larger, so this pins the rounding mode as well as the rounding step itself."""
    levels = {r[0]: (float(r[2]), float(r[3])) for r in _read_table("lab_error_levels.txt")}
    want_max, want_fro = levels["f16_in_f32_acc"]
    n = 1024
    A = synth.matrix(n, n, seed=0, tensor=0, dist="unit")
    B = synth.matrix(n, n, seed=0, tensor=1, dist="unit")
    ref = A.astype(np.float64) @ B.astype(np.float64)
    D, _ = oracle_mod.gemm(A, B, None, 1.0, 0.0, f16_inputs=True, want_mag=False)
    e_max, e_fro = _errors(D, ref)
    assert want_fro / 1.5 <= e_fro <= want_fro * 1.5, e_fro
    assert want_max / 2.0 <= e_max <= want_max * 2.0, e_max
    # the same statistic for truncated operands falls far outside the band
    trunc = lambda x: (x.view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)
    Dt = (trunc(A).astype(np.float64) @ trunc(B).astype(np.float64)).astype(np.float32)
    assert _errors(Dt, ref)[1] > 5 * want_fro
    # and without the rounding step the error is at the f32 level, far below the band
    D32, _ = oracle_mod.gemm(A, B, None, 1.0, 0.0, f16_inputs=False, want_mag=False)
    assert _errors(D32, ref)[1] < want_fro / 50


# ----------------------------------------------------------------------------------------
# f64 -> f16 in one rounding, and the GEMM with an f16 result (the lab's cuBLAS f16 GEMM,
# Part 4 "precision": f16 operands and output, f32 accumulation)
# ----------------------------------------------------------------------------------------

def _np_f16_bits_from_f64(x):
    # numpy converts float64 to binary16 directly, rounding to nearest with ties to even
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def test_f64_to_f16_golden_cases(oracle_mod):
    cases = [
        (0.0, 0x0000), (-0.0, 0x8000), (1.0, 0x3C00), (-2.0, 0xC000),
        (65504.0, 0x7BFF),                       # largest finite
        (65519.99999999999, 0x7BFF),             # just below the overflow tie
        (65520.0, 0x7C00),                       # the tie rounds to even: infinity
        (1e300, 0x7C00), (-1e300, 0xFC00), (float("inf"), 0x7C00),
        (2.0 ** -24, 0x0001),                    # smallest subnormal
        (2.0 ** -25, 0x0000),                    # tie between 0 and 2^-24: even is 0
        (3 * 2.0 ** -25, 0x0002),                # tie between 1 and 2 units: even is 2
        (2.0 ** -25 + 2.0 ** -60, 0x0001),       # just above the tie: an f32 step would lose it
        (2.0 ** -14 - 2.0 ** -26, 0x0400),       # rounds up into the smallest normal
        (1.0 + 2.0 ** -11, 0x3C00),              # tie at 1: even
        (1.0 + 3 * 2.0 ** -11, 0x3C02),          # tie at 1 + 2^-10: even is 1 + 2^-9
        (1.0 + 2.0 ** -11 + 2.0 ** -40, 0x3C01), # a float64 tail an f32 rounding would drop
        (2047.0, 0x67FF), (2047.5, 0x6800),      # tie between 2047 and 2048: even is 2048
        (2048.5, 0x6800), (2049.0, 0x6800), (2051.0, 0x6802),
        (1e-300, 0x0000), (-1e-300, 0x8000),
    ]
    for x, want in cases:
        got = int(oracle_mod.f64_to_f16_bits(np.array([x]))[0])
        assert got == want, (x, hex(got), hex(want))
    assert (int(oracle_mod.f64_to_f16_bits(np.array([float("nan")]))[0]) & 0x7FFF) > 0x7C00


def test_f64_to_f16_matches_numpy(oracle_mod):
    rng = np.random.default_rng(11)
    # magnitudes across the subnormal, normal and overflow ranges, both signs
    mags = np.ldexp(rng.uniform(1.0, 2.0, 20000), rng.integers(-30, 18, 20000))
    x = mags * rng.choice([-1.0, 1.0], 20000)
    # exact ties at every spacing: (2q + 1) / 2 units of 2^-24 .. 2^5
    q = rng.integers(0, 2048, 4000)
    sp = rng.integers(-24, 6, 4000)
    ties = np.ldexp(2.0 * q + 1.0, sp - 1)
    allx = np.concatenate([x, ties, -ties])
    got = oracle_mod.f64_to_f16_bits(allx)
    want = _np_f16_bits_from_f64(allx)
    bad = np.nonzero(~_same_f16(got, want))[0]
    assert bad.size == 0, [(float(allx[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]


@pytest.mark.parametrize("f16", [False, True])
def test_gemm_f16out_integer_inputs(oracle_mod, f16):
    # integer operands: the float64 sum is exact, and results between 2048 and 65504 land on
    # the f16 grid's even-spaced integers, so the rounding of exact values is what is checked
    rng = np.random.default_rng(3)
    M, N, K = 24, 40, 300
    A = rng.integers(-3, 4, (M, K)).astype(np.float32)
    B = rng.integers(-3, 4, (K, N)).astype(np.float32)
    C = rng.integers(-50, 51, (M, N)).astype(np.float32)
    reached = False
    for alpha, beta in ((1.0, 0.0), (48.0, 0.5), (-24.5, 2.0), (0.0, 1.5)):
        D16, _ = oracle_mod.gemm_f16out(A, B, C, alpha, beta, f16_inputs=f16)
        exact = alpha * (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64) + beta * C.astype(np.float64)
        assert np.array_equal(D16, _np_f16_bits_from_f64(exact)), (alpha, beta)
        reached |= bool(((np.abs(exact) > 2048) & (np.abs(exact) < 65504)).any())
    assert reached   # the test reaches the spaced-out integers


def test_gemm_f16out_brute_force_exact_rationals(oracle_mod):
    rnd = random.Random(17)
    for trial in range(60):
        M, N, K = rnd.randint(1, 4), rnd.randint(1, 4), rnd.randint(1, 6)
        # f16 operands with full 11-bit significands at mixed scales
        A = (synth.matrix(M, K, seed=300 + trial, tensor=0) * 4).astype(np.float16).astype(np.float32)
        B = (synth.matrix(K, N, seed=300 + trial, tensor=1) * 64).astype(np.float16).astype(np.float32)
        C = synth.matrix(M, N, seed=300 + trial, tensor=2).astype(np.float16).astype(np.float32)
        alpha = rnd.choice([1.0, -0.5, 3.0, 0.375])
        beta = rnd.choice([0.0, 1.0, -2.0, 0.25])
        D16, _ = oracle_mod.gemm_f16out(A, B, C, alpha, beta)
        for i in range(M):
            for j in range(N):
                s = sum(Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(K))
                exact = Fraction(alpha) * s + Fraction(beta) * Fraction(float(C[i, j]))
                # the exact value needs at most 53 significant bits here, so float() is exact
                assert Fraction(float(exact)) == exact
                want = int(_np_f16_bits_from_f64(np.array([float(exact)]))[0])
                assert int(D16[i, j]) == want, (trial, i, j, float(exact))


def test_gemm_f16out_agrees_with_gemm_where_f32_is_exact(oracle_mod):
    # on f16-grid data whose results are exact in f32, rounding the f32 result to f16 and
    # rounding straight from float64 agree
    A = synth.matrix(17, 23, seed=5, tensor=0, dist="int3")
    B = synth.matrix(23, 9, seed=5, tensor=1, dist="int3")
    C = synth.matrix(17, 9, seed=5, tensor=2, dist="int3")
    D32, _ = oracle_mod.gemm(A, B, C, 0.5, -1.0)
    D16, _ = oracle_mod.gemm_f16out(A, B, C, 0.5, -1.0)
    assert np.array_equal(D16, _np_f16_bits(D32))
