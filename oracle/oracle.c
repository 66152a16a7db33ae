/*
 * oracle.c -- the CPU oracle for C = alpha * A @ B + beta * C.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct reference that the
 * CUDA path is checked against.  Only the tests, the smoke check and the benchmark's CPU
 * baseline load it; the product library never links, calls or falls back to it, and it
 * shares no code, header or table with the CUDA sources.
 *
 * What it computes (cited to the pages it follows):
 *
 *   "gemm, f32" (phobos-lang.dev/docs/examples/gemm-fp32/), the kernel listing and
 *   section "The epilogue": an accumulator tile starts at zero, the k loop adds the
 *   product of A's and B's panels into it, and the epilogue stores alpha * acc + beta * c_old
 *   over the same tile of C.  Written out per element, that is
 *
 *       acc_ij = sum_{k=0}^{K-1} a_ik * b_kj              (float64, k ascending)
 *       C'_ij  = round_to_f32(alpha * acc_ij + beta * C_ij)  (float64, one final rounding)
 *
 *   "gemm on tensor cores" (phobos-lang.dev/docs/examples/gemm-fp16tc-fp32acc/), section
 *   "What changes": the operands are rounded to f16 and the products summed in f32, so the
 *   rounding costs precision in the inputs and not in the sums.  The oracle therefore rounds
 *   every element of A and B to the nearest f16 (ties to even, the IEEE 754 default; the
 *   page only says "rounded") and then runs the same float64 sum.  f16*f16 and f32*f32
 *   products are exact in float64, so the only rounding inside the sum is float64
 *   addition, with relative error at most K * 2^-53.
 *
 *   "Matrix Multiplication: The Operation Behind Modern AI" (lenatriestounderstand.com,
 *   .../002-matrix-multiplication/lab), Part 2: every kernel there is compared with a
 *   float64 product of the same inputs; this oracle is that float64 product, plus alpha,
 *   beta and C.
 *
 *   The same lab, Part 4 ("precision") and Part 5, times cuBLAS's f16 GEMM: f16 operands
 *   and an f16 result, accumulated in f32.  oracle_gemm_f16out is that product's
 *   definition: the float64 sum and epilogue as above, then one rounding straight to f16
 *   (to nearest, ties to even) instead of to f32.
 *
 * Readings of points the pages leave open:
 *   - beta == 0: C is not read (the BLAS reading), so NaN in C does not propagate.
 *   - alpha == 0: A and B are not read; C' = round(beta * C).
 *   - K == 0: acc = 0, so C' = round(beta * C).
 *   - f16 rounding: round to nearest, ties to even, subnormals kept, |x| >= 65520 -> inf,
 *     NaN stays NaN (quiet), as IEEE 754 binary16.
 *
 * Build: plain C99; OpenMP over rows when the compiler has it.  Build with
 * -ffp-contract=off so that no multiply-add is fused and the result is the same on every
 * host.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------------------ */
/* f32 -> f16, round to nearest with ties to even, from the binary32 / binary16 formats.  */
/* binary32: 1 sign, 8 exponent (bias 127), 23 fraction bits.                            */
/* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits; the smallest subnormal is    */
/* 2^-24 and the largest finite value 65504.                                              */
/* ------------------------------------------------------------------------------------ */

/* Round the non-negative integer `v` right by `s` bits (1 <= s <= 31), to nearest, ties to
 * the even result. */
static uint32_t shift_round_even(uint32_t v, int s) {
    uint32_t q = v >> s;
    uint32_t rem = v & ((1u << s) - 1u);
    uint32_t half = 1u << (s - 1);
    if (rem > half || (rem == half && (q & 1u))) q += 1u;
    return q;
}

uint16_t oracle_f32_to_f16_bits(float f) {
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    uint32_t sign = (x >> 16) & 0x8000u;
    int exp32 = (int)((x >> 23) & 0xFFu);
    uint32_t frac = x & 0x7FFFFFu;

    if (exp32 == 0xFF) {                       /* inf or NaN */
        if (frac == 0) return (uint16_t)(sign | 0x7C00u);
        return (uint16_t)(sign | 0x7E00u | (frac >> 13));   /* quiet NaN, top payload bits */
    }
    if (exp32 == 0) {                          /* zero or f32 subnormal: |x| < 2^-126 */
        return (uint16_t)sign;                 /* far below half of 2^-24: rounds to zero */
    }
    /* |x| = m * 2^(exp32 - 150) with m the 24-bit significand including the hidden bit. */
    uint32_t m = frac | 0x800000u;
    int e16 = exp32 - 127 + 15;                /* biased f16 exponent if x is f16-normal */

    if (e16 >= 31) return (uint16_t)(sign | 0x7C00u);       /* |x| >= 65536: overflow */

    if (e16 <= 0) {
        /* f16 subnormal range: the result is an integer count q of 2^-24 units,
         * q = round(m * 2^(exp32 - 150 + 24)) = round(m >> (126 - exp32)). */
        int s = 126 - exp32;                   /* >= 14 here */
        if (s >= 32) return (uint16_t)sign;    /* m < 2^24 <= half of 2^s: rounds to zero */
        uint32_t q = shift_round_even(m, s);   /* q == 0x400 is the smallest normal: right */
        return (uint16_t)(sign | q);
    }
    /* f16 normal: keep 10 fraction bits, round the 13 dropped ones.  A carry out of the
     * fraction moves into the exponent, and out of the largest exponent gives 0x7C00 (inf),
     * which is the correct rounding of 65520 <= |x| < 65536. */
    uint32_t q = ((uint32_t)e16 << 10) | (frac >> 13);
    uint32_t rem = frac & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (q & 1u))) q += 1u;
    return (uint16_t)(sign | q);
}

float oracle_f16_bits_to_f32(uint16_t h) {
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    int e = (h >> 10) & 0x1F;
    uint32_t frac = h & 0x3FFu;
    float out;
    if (e == 0x1F) {
        uint32_t bits = sign | 0x7F800000u | (frac << 13);
        memcpy(&out, &bits, sizeof out);
        return out;
    }
    /* value = (e == 0 ? frac : 1024 + frac) * 2^(max(e,1) - 25); exact in float64 and f32 */
    double mag = (e == 0) ? ldexp((double)frac, -24) : ldexp((double)(1024u + frac), e - 25);
    out = (float)mag;
    return sign ? -out : out;
}

/* f64 -> f16, round to nearest with ties to even, in one step (no intermediate f32).
 * |x| lies in [2^e, 2^(e+1)); the f16 spacing there is 2^(e-10) for e >= -14 (normal) and
 * 2^-24 below (subnormal).  x / spacing is rounded to an integer q, ties to even; q = 2048
 * (normal) carries into the exponent, q = 1024 (subnormal) is the smallest normal, and an
 * exponent past 15 is infinity.  Scaling by a power of two is exact in float64. */
uint16_t oracle_f64_to_f16_bits(double x) {
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
    const double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7C00u);
    if (a == 0.0) return sign;
    int fe;
    (void)frexp(a, &fe);                       /* a = m * 2^fe, 0.5 <= m < 1 */
    const int e = fe - 1;                      /* 2^e <= a < 2^(e+1) */
    const int spacing = e < -14 ? -24 : e - 10;
    const double scaled = ldexp(a, -spacing);  /* exact */
    const double fl = floor(scaled);
    const double rem = scaled - fl;            /* exact */
    if (fl >= 4096.0) return (uint16_t)(sign | 0x7C00u);    /* only when e > 15 */
    uint32_t q = (uint32_t)fl;
    if (rem > 0.5 || (rem == 0.5 && (q & 1u))) q += 1u;
    if (e < -14) return (uint16_t)(sign | q);  /* q <= 1024: 1024 is the smallest normal */
    int be = e + 15;                           /* biased exponent, >= 1 */
    if (q == 2048u) { q = 1024u; be += 1; }
    if (be >= 31) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | ((uint32_t)be << 10) | (q - 1024u));
}

void oracle_f32_to_f16(const float* x, uint16_t* h, int64_t n) {
    for (int64_t i = 0; i < n; ++i) h[i] = oracle_f32_to_f16_bits(x[i]);
}

/* y[i] = the value of x[i] after rounding to f16, held exactly in an f32. */
void oracle_round_f16(const float* x, float* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_f16_bits_to_f32(oracle_f32_to_f16_bits(x[i]));
}

/* ------------------------------------------------------------------------------------ */
/* The GEMM.                                                                             */
/* ------------------------------------------------------------------------------------ */

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Row i of the result: D[i, :] and, if mag_out is not NULL, sum_k |a_ik| |b_kj| for the
 * error bound.  `a` is row i of A (length K), already rounded if the f16 variant asked.
 * The one final rounding of alpha * acc + beta * c goes to f32 (d) or, when d16 is not
 * NULL, straight from float64 to f16 bits (d16). */
static void gemm_row(int64_t N, int64_t K, double alpha, const float* a, const float* B,
                     double beta, const float* c, float* d, uint16_t* d16, double* mag_out,
                     double* acc, double* mag) {
    for (int64_t j = 0; j < N; ++j) { acc[j] = 0.0; if (mag) mag[j] = 0.0; }
    if (alpha != 0.0) {
        for (int64_t k = 0; k < K; ++k) {
            const double aik = (double)a[k];
            const float* brow = B + k * N;
            for (int64_t j = 0; j < N; ++j) acc[j] += aik * (double)brow[j];
            if (mag) {
                const double aabs = fabs(aik);
                for (int64_t j = 0; j < N; ++j) mag[j] += aabs * fabs((double)brow[j]);
            }
        }
    }
    for (int64_t j = 0; j < N; ++j) {
        double v = alpha * acc[j];
        if (beta != 0.0) v += beta * (double)c[j];
        if (d16)
            d16[j] = oracle_f64_to_f16_bits(v);
        else
            d[j] = (float)v;
        if (mag_out) mag_out[j] = mag ? mag[j] : 0.0;
    }
}

/*
 * D = round_f32(alpha * (A @ B) + beta * C), every array row-major and contiguous:
 * A is M x K, B is K x N, C and D are M x N.  D may equal C (in place).  If mag is not
 * NULL it receives sum_k |a_ik| |b_kj| (float64, M x N).  round_inputs_f16 != 0 selects the
 * tensor-core variant: A and B are rounded to f16 (to nearest, ties to even) first.
 * Returns 0, or -1 if memory ran out or a size is negative.
 */
static int gemm_impl(int64_t M, int64_t N, int64_t K, float alpha, const float* A, const float* B,
                     float beta, const float* C, float* D, uint16_t* D16, double* mag,
                     int round_inputs_f16) {
    if (M < 0 || N < 0 || K < 0) return -1;
    if (M == 0 || N == 0) return 0;
    const double a64 = (double)alpha, b64 = (double)beta;
    const float* Ause = A;
    const float* Buse = B;
    float* Ar = NULL;
    float* Br = NULL;
    if (round_inputs_f16 && a64 != 0.0 && K > 0) {
        Ar = (float*)malloc(sizeof(float) * (size_t)(M * K));
        Br = (float*)malloc(sizeof(float) * (size_t)(K * N));
        if (!Ar || !Br) { free(Ar); free(Br); return -1; }
        oracle_round_f16(A, Ar, M * K);
        oracle_round_f16(B, Br, K * N);
        Ause = Ar;
        Buse = Br;
    }
    int failed = 0;
#pragma omp parallel
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)N);
        double* mg = mag ? (double*)malloc(sizeof(double) * (size_t)N) : NULL;
        if (!acc || (mag && !mg)) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < M; ++i) {
                gemm_row(N, K, a64, Ause + i * K, Buse, b64, C ? C + i * N : NULL, D ? D + i * N : NULL,
                         D16 ? D16 + i * N : NULL, mag ? mag + i * N : NULL, acc, mg);
            }
        }
        free(acc);
        free(mg);
    }
    free(Ar);
    free(Br);
    return failed ? -1 : 0;
}

int oracle_gemm(int64_t M, int64_t N, int64_t K, float alpha, const float* A, const float* B,
                float beta, const float* C, float* D, double* mag, int round_inputs_f16) {
    return gemm_impl(M, N, K, alpha, A, B, beta, C, D, NULL, mag, round_inputs_f16);
}

/*
 * The same product with an f16 result, as a GEMM with half-precision output computes it:
 * D16 = round_f16(alpha * (A @ B) + beta * C) with one rounding, straight from float64 (the
 * values of A, B and C are given as f32; for half-precision operands they are f16 values
 * held exactly).  mag and round_inputs_f16 as in oracle_gemm.
 */
int oracle_gemm_f16out(int64_t M, int64_t N, int64_t K, float alpha, const float* A, const float* B,
                       float beta, const float* C, uint16_t* D16, double* mag, int round_inputs_f16) {
    return gemm_impl(M, N, K, alpha, A, B, beta, C, NULL, D16, mag, round_inputs_f16);
}

/*
 * The same definition, evaluated only at the n positions (rows[t], cols[t]): out[t] is
 * round_f32(alpha * sum_k a_ik b_kj + beta * C_ij) with k ascending in float64, and mag[t]
 * (if not NULL) is sum_k |a_ik| |b_kj|.  Used to check single outputs of problems too large
 * to evaluate whole.  Returns 0, or -1 on a bad index.
 */
int oracle_gemm_at(int64_t M, int64_t N, int64_t K, float alpha, const float* A, const float* B,
                   float beta, const float* C, const int64_t* rows, const int64_t* cols,
                   int64_t n, float* out, double* mag, int round_inputs_f16) {
    int bad = 0;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        const int64_t i = rows[t], j = cols[t];
        if (i < 0 || i >= M || j < 0 || j >= N) {
#pragma omp atomic write
            bad = 1;
            continue;
        }
        double acc = 0.0, mg = 0.0;
        if (alpha != 0.0f) {
            for (int64_t k = 0; k < K; ++k) {
                double a = (double)A[i * K + k];
                double b = (double)B[k * N + j];
                if (round_inputs_f16) {
                    a = (double)oracle_f16_bits_to_f32(oracle_f32_to_f16_bits((float)a));
                    b = (double)oracle_f16_bits_to_f32(oracle_f32_to_f16_bits((float)b));
                }
                acc += a * b;
                mg += fabs(a) * fabs(b);
            }
        }
        double v = (double)alpha * acc;
        if (beta != 0.0f) v += (double)beta * (double)C[i * N + j];
        out[t] = (float)v;
        if (mag) mag[t] = mg;
    }
    return bad ? -1 : 0;
}
