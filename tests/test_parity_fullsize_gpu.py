"""Parity at the workloads' full sizes, in the launch configuration the benchmark uses
(no pinned configuration), through the C ABI.

Integer-valued inputs are compared with the oracle bit for bit over the whole result at
4096^3 and at the masked (4095, 4097, 4093); everywhere else outputs are sampled (random
positions plus every tile-edge row and column) and each sample is evaluated on its own by
the oracle's single-element routine.
"""
import numpy as np
import pytest

import oracle
from dense_gemm_04_gb300 import phx, synth
from tests.gpu_util import VARIANTS, assert_bits_equal, assert_within_bound, run_cuda

pytestmark = pytest.mark.gpu

SHAPES = [
    # (M, N, K, alpha, beta)
    (4096, 4096, 4096, 1.0, 0.5),      # the headline f32 and f16-TC configurations
    (8192, 8192, 1024, 2.0, -1.0),     # shape / alignment sweep
    (1024, 1024, 16384, 2.0, -1.0),
    (16384, 128, 4096, 2.0, -1.0),
    (4095, 4097, 4093, 2.0, -1.0),     # masked edges in every dimension
    (512, 512, 512, 1.0, 0.0),         # arithmetic-intensity sweep
    (1024, 1024, 1024, 1.0, 0.0),
    (2048, 2048, 2048, 1.0, 0.0),
    (8192, 8192, 8192, 1.0, 0.0),
    (16384, 16384, 16384, 1.0, 0.0),
]


def _sample_positions(M, N, n=2048, seed=0):
    rng = np.random.default_rng(seed)
    rows = list(rng.integers(0, M, n))
    cols = list(rng.integers(0, N, n))
    edge_r = sorted({r for t in range(0, M, 128) for r in (t, t + 127) if r < M} | {M - 1})
    edge_c = sorted({c for t in range(0, N, 64) for c in (t, t + 63) if c < N} | {N - 1})
    for r in edge_r[:: max(1, len(edge_r) // 64)]:
        rows.append(r); cols.append(int(rng.integers(0, N)))
    for c in edge_c[:: max(1, len(edge_c) // 64)]:
        rows.append(int(rng.integers(0, M))); cols.append(c)
    return np.array(rows, np.int64), np.array(cols, np.int64)


@pytest.mark.parametrize("vname", list(VARIANTS))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s[:3])))
def test_fullsize_sampled(vname, shape):
    M, N, K, alpha, beta = shape
    variant, f16 = VARIANTS[vname]
    dists = ["uniform"] if M * N * K > 2 ** 40 else ["uniform", "int3"]
    for dist in dists:
        A, B, C = synth.problem(M, N, K, seed=0, dist=dist)
        st, got = run_cuda(variant, A, B, C, alpha, beta)
        assert st == phx.PHX_OK, phx.status_string(st)
        rows, cols = _sample_positions(M, N)
        want, mag = oracle.gemm_at(A, B, C, alpha, beta, rows, cols, f16_inputs=f16)
        g = got[rows, cols]
        what = f"{vname} {shape[:3]} {dist} [{phx.get_config(variant, M, N, K)}]"
        if dist == "int3":
            assert_bits_equal(g, want, what)
        else:
            assert_within_bound(g, want, mag, C[rows, cols], K, alpha, beta, what)


@pytest.mark.parametrize("vname", list(VARIANTS))
@pytest.mark.parametrize("shape", [(4096, 4096, 4096, 1.0, 0.5), (4095, 4097, 4093, 2.0, -1.0)],
                         ids=["4096^3", "4095x4097x4093"])
def test_fullsize_integer_bit_exact_everywhere(vname, shape):
    M, N, K, alpha, beta = shape
    variant, f16 = VARIANTS[vname]
    A, B, C = synth.problem(M, N, K, seed=1, dist="int3")
    st, got = run_cuda(variant, A, B, C, alpha, beta)
    assert st == phx.PHX_OK
    want, _ = oracle.gemm(A, B, C, alpha, beta, f16_inputs=f16, want_mag=False)
    assert_bits_equal(got, want, f"{vname} {shape[:3]}")
