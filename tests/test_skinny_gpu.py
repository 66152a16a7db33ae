"""The skinny kernel (few rows of A; the matrix-multiplication lab's skinny-matrix sweep,
Part 5), both precisions, through the C ABI on a GB300, against the oracle.

It is the default for small M, and for few columns against many rows with A stored M x K (as
the transposed product, streaming A's rows), and can be pinned ("SKINNY") for any M.  Covered
here: few columns (1 to 8, ragged, long and short K, every storage order); M from
1 to 64 at the sweep's K = N = 4096 in both precisions; ragged N (scalar loads, partial
column strips), K shorter than one slice and K split into many slices; A stored transposed
(read in place); B stored transposed (N x K, the layout of W in x @ W^T: the kernel that
streams B's rows), from 1 to 64 rows, ragged and long K, aligned or not; a B pointer only
4-byte aligned; M beyond one block of 16 rows; the degenerate cases; run-to-run determinism.
"""
import numpy as np
import pytest

import oracle
from dense_gemm_04_gb300 import phx, synth
from tests.gpu_util import VARIANTS, assert_bits_equal, assert_within_bound, run_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _pin_skinny():
    for v in (phx.VARIANT_SGEMM, phx.VARIANT_F16TC):
        phx.set_config(v, "SKINNY")
    yield
    for v in (phx.VARIANT_SGEMM, phx.VARIANT_F16TC):
        phx.set_config(v, None)
    assert phx.check_device_status() == phx.PHX_OK


def _check(vname, M, N, K, alpha, beta, dist, seed=0):
    variant, f16 = VARIANTS[vname]
    A, B, C = synth.problem(M, N, K, seed=seed, dist=dist)
    want, mag = oracle.gemm(A, B, C, alpha, beta, f16_inputs=f16)
    st, got = run_cuda(variant, A, B, C, alpha, beta)
    assert st == phx.PHX_OK, phx.status_string(st)
    what = f"skinny {vname} {(M, N, K)} {dist}"
    if dist == "int3":
        assert_bits_equal(got, want, what)
    else:
        assert_within_bound(got, want, mag, C, K, alpha, beta, what)
    return got


@pytest.mark.parametrize("vname", list(VARIANTS))
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 13, 16, 17, 32, 33, 64])
def test_skinny_sweep_shapes(vname, M):
    # the lab's sweep: K = N = 4096
    _check(vname, M, 4096, 4096, 1.0, 0.0, "int3", seed=M)
    _check(vname, M, 4096, 4096, 2.0, -1.0, "uniform", seed=M)


@pytest.mark.parametrize("vname", list(VARIANTS))
@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 7), (7, 4095, 300), (16, 130, 513), (2, 129, 12345),
                                   (9, 1, 4096), (4, 4100, 64), (64, 200, 8), (20, 384, 1000)])
def test_skinny_ragged(vname, shape):
    M, N, K = shape
    _check(vname, M, N, K, 1.5, 0.5, "int3", seed=1)
    _check(vname, M, N, K, 1.5, 0.5, "uniform", seed=2)


@pytest.mark.parametrize("vname", list(VARIANTS))
def test_skinny_large_m(vname):
    # any M, as blocks of 16 rows (the pinned configuration of every test of the suite)
    _check(vname, 301, 263, 197, 2.0, -1.0, "int3")
    _check(vname, 256, 256, 256, 1.5, 0.5, "uniform")


@pytest.mark.parametrize("vname", list(VARIANTS))
def test_skinny_transposed_operands(vname):
    import torch
    variant, f16 = VARIANTS[vname]
    fn = phx.phx_sgemm_ex if variant == phx.VARIANT_SGEMM else phx.phx_gemm_f16tc_f32acc_ex
    for M, N, K in ((1, 4096, 4096), (13, 333, 777)):
        A, B, C = synth.problem(M, N, K, seed=9, dist="int3")
        want, _ = oracle.gemm(A, B, C, 1.0, 1.0, f16_inputs=f16)
        for op_a in (phx.OP_N, phx.OP_T):
            for op_b in (phx.OP_N, phx.OP_T):
                a = np.ascontiguousarray(A.T if op_a == phx.OP_T else A)
                b = np.ascontiguousarray(B.T if op_b == phx.OP_T else B)
                dA, dB = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
                dC = torch.from_numpy(C.copy()).cuda()
                st = fn(op_a, op_b, M, N, K, 1.0, dA.data_ptr(), dB.data_ptr(), 1.0, dC.data_ptr(),
                        torch.cuda.current_stream().cuda_stream)
                torch.cuda.synchronize()
                assert st == phx.PHX_OK
                assert_bits_equal(dC.cpu().numpy(), want, f"{vname} ops ({op_a},{op_b}) {(M, N, K)}")


def _run_ex(variant, op_a, op_b, A, B, C, alpha, beta, offset=0):
    import torch
    M, K = A.shape
    N = B.shape[1]

    def dev(x):
        flat = torch.zeros(x.size + offset, dtype=torch.float32)
        flat[offset:] = torch.from_numpy(np.ascontiguousarray(x).reshape(-1))
        return flat.cuda()

    a = A.T if op_a == phx.OP_T else A
    b = B.T if op_b == phx.OP_T else B
    dA, dB = dev(a), dev(b)
    dC = torch.from_numpy(C.copy()).cuda()
    fn = phx.phx_sgemm_ex if variant == phx.VARIANT_SGEMM else phx.phx_gemm_f16tc_f32acc_ex
    st = fn(op_a, op_b, M, N, K, alpha, dA.data_ptr() + 4 * offset, dB.data_ptr() + 4 * offset, beta,
            dC.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return st, dC.cpu().numpy()


@pytest.mark.parametrize("vname", list(VARIANTS))
@pytest.mark.parametrize("shape", [(1, 4096, 4096), (2, 4096, 4096), (4, 4096, 4096), (8, 4096, 4096),
                                   (16, 4096, 4096), (33, 4096, 4096), (3, 333, 777), (16, 33, 130),
                                   (2, 100, 65536), (5, 1, 64), (1, 1, 1), (64, 64, 4100)])
def test_skinny_b_stored_transposed(vname, shape):
    # B stored N x K (x @ W^T): the kernel that streams B's rows
    variant, f16 = VARIANTS[vname]
    M, N, K = shape
    for dist, seed in (("int3", 21), ("uniform", 22)):
        A, B, C = synth.problem(M, N, K, seed=seed, dist=dist)
        want, mag = oracle.gemm(A, B, C, 2.0, -1.0, f16_inputs=f16)
        for op_a in (phx.OP_N, phx.OP_T):
            st, got = _run_ex(variant, op_a, phx.OP_T, A, B, C, 2.0, -1.0)
            assert st == phx.PHX_OK, phx.status_string(st)
            what = f"skinny {vname} B^T {shape} {dist} op_a={op_a}"
            if dist == "int3":
                assert_bits_equal(got, want, what)
            else:
                assert_within_bound(got, want, mag, C, K, 2.0, -1.0, what)
    # W only 4-byte aligned: 4-byte copies
    A, B, C = synth.problem(M, N, K, seed=23, dist="int3")
    want, _ = oracle.gemm(A, B, C, 1.0, 0.5, f16_inputs=f16)
    st, got = _run_ex(variant, phx.OP_N, phx.OP_T, A, B, C, 1.0, 0.5, offset=1)
    assert st == phx.PHX_OK
    assert_bits_equal(got, want, f"skinny {vname} B^T {shape} unaligned")


@pytest.mark.parametrize("vname", list(VARIANTS))
def test_skinny_unaligned_b(vname):
    import torch
    variant, f16 = VARIANTS[vname]
    M, N, K = 6, 1024, 1024
    A, B, C = synth.problem(M, N, K, seed=10, dist="int3")
    want, _ = oracle.gemm(A, B, C, 1.0, 0.0, f16_inputs=f16)
    flat = torch.zeros(K * N + 1)
    flat[1:] = torch.from_numpy(B.reshape(-1))
    dB = flat.cuda()
    dA = torch.from_numpy(A).cuda()
    dC = torch.zeros(M, N, device="cuda")
    fn = phx.phx_sgemm if variant == phx.VARIANT_SGEMM else phx.phx_gemm_f16tc_f32acc
    st = fn(M, N, K, 1.0, dA.data_ptr(), dB.data_ptr() + 4, 0.0, dC.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == phx.PHX_OK
    assert_bits_equal(dC.cpu().numpy(), want, f"{vname} unaligned B")


@pytest.mark.parametrize("vname", list(VARIANTS))
def test_skinny_degenerate_and_special_values(vname):
    variant, f16 = VARIANTS[vname]
    M, N, K = 4, 300, 600
    A, B, C = synth.problem(M, N, K, seed=11, dist="int3")
    # beta == 0 with NaN in C: C is not read
    st, got = run_cuda(variant, A, B, np.full_like(C, np.nan), 1.0, 0.0)
    want, _ = oracle.gemm(A, B, C, 1.0, 0.0, f16_inputs=f16)
    assert st == phx.PHX_OK
    assert_bits_equal(got, want, "beta = 0, C = NaN")
    # an Inf in row 0 of A reaches row 0 of C only
    A2 = A.copy()
    A2[0, 5] = np.inf
    B2 = np.abs(B) + 1
    st, got = run_cuda(variant, A2, B2, C, 1.0, 0.0)
    assert st == phx.PHX_OK
    assert np.isinf(got[0]).all() and np.isfinite(got[1:]).all()
    # f16 variant: values beyond the f16 range round to infinity, as the pages' rounding does
    if f16:
        A3 = np.zeros((1, 1), np.float32)
        A3[0, 0] = 70000.0
        B3 = np.ones((1, 3), np.float32)
        st, got = run_cuda(variant, A3, B3, np.zeros((1, 3), np.float32), 1.0, 0.0)
        assert st == phx.PHX_OK and np.isinf(got).all()


@pytest.mark.parametrize("vname", list(VARIANTS))
def test_skinny_is_deterministic(vname):
    variant, _ = VARIANTS[vname]
    A, B, C = synth.problem(24, 4096, 4096, seed=12, dist="uniform")
    _, r1 = run_cuda(variant, A, B, C, 1.0, 0.5)
    _, r2 = run_cuda(variant, A, B, C, 1.0, 0.5)
    assert_bits_equal(r1, r2, "two runs")


@pytest.mark.parametrize("vname", list(VARIANTS))
@pytest.mark.parametrize("shape", [(4096, 1, 4096), (2085, 7, 2050), (1030, 8, 333), (1024, 3, 65536),
                                   (1500, 5, 3000), (5000, 2, 64)])
def test_few_columns_transposed_product(vname, shape):
    # few columns against many rows: C^T = B^T @ A^T on the kernel that streams rows (of A
    # here), C^T written transposed.  Ragged M and K; K % 4 != 0 (A's rows not on 16 bytes);
    # K split across a cluster, and into planes at K = 65536; one chunk of K.
    M, N, K = shape
    _check(vname, M, N, K, 1.5, 0.5, "int3", seed=31)
    _check(vname, M, N, K, 2.0, -1.0, "uniform", seed=32)
    # beta = 0 with NaN in C: C is not read
    variant, f16 = VARIANTS[vname]
    A, B, C = synth.problem(M, N, K, seed=33, dist="int3")
    want, _ = oracle.gemm(A, B, C, 1.0, 0.0, f16_inputs=f16)
    st, got = run_cuda(variant, A, B, np.full_like(C, np.nan), 1.0, 0.0)
    assert st == phx.PHX_OK
    assert_bits_equal(got, want, f"{vname} few columns {shape}, beta = 0")


@pytest.mark.parametrize("vname", list(VARIANTS))
def test_few_columns_storage_orders(vname):
    # B stored N x K (plain rows of the few-row operand) and A stored at a 4-byte offset (its
    # rows copied 4 bytes at a time) take the transposed product; A stored K x M takes the
    # rows of A in blocks of 16 instead.  All against the oracle.
    variant, f16 = VARIANTS[vname]
    M, N, K = 1500, 5, 3000
    A, B, C = synth.problem(M, N, K, seed=34, dist="int3")
    want, _ = oracle.gemm(A, B, C, 1.0, 0.5, f16_inputs=f16)
    for op_a, op_b, off in ((phx.OP_N, phx.OP_T, 0), (phx.OP_N, phx.OP_N, 1), (phx.OP_N, phx.OP_T, 1),
                            (phx.OP_T, phx.OP_N, 0), (phx.OP_T, phx.OP_T, 0)):
        st, got = _run_ex(variant, op_a, op_b, A, B, C, 1.0, 0.5, offset=off)
        assert st == phx.PHX_OK, phx.status_string(st)
        assert_bits_equal(got, want, f"{vname} few columns ops ({op_a},{op_b}) offset {off}")


def test_default_routes_few_columns_to_skinny():
    for v in (phx.VARIANT_SGEMM, phx.VARIANT_F16TC):
        phx.set_config(v, None)
    assert phx.get_config(phx.VARIANT_SGEMM, 4096, 16, 4096) == "SKINNY"
    assert phx.get_config(phx.VARIANT_F16TC, 4096, 4, 4096) == "SKINNY"
    assert phx.get_config(phx.VARIANT_F16TC, 4096, 8, 4096) != "SKINNY"
    for vname, n in (("sgemm", 16), ("f16tc", 4)):
        _check(vname, 4096, n, 4096, 1.0, 0.5, "int3", seed=35)
        assert phx.last_config(VARIANTS[vname][0]) == "SKINNY"
    # A stored K x M: the default tile instead
    variant, f16 = VARIANTS["sgemm"]
    A, B, C = synth.problem(2048, 4, 2048, seed=36, dist="int3")
    want, _ = oracle.gemm(A, B, C, 1.0, 0.5, f16_inputs=f16)
    st, got = _run_ex(variant, phx.OP_T, phx.OP_N, A, B, C, 1.0, 0.5)
    assert st == phx.PHX_OK
    assert phx.last_config(variant) != "SKINNY"
    assert_bits_equal(got, want, "few columns, A stored K x M")


def test_default_routes_small_m_to_skinny():
    for v in (phx.VARIANT_SGEMM, phx.VARIANT_F16TC):
        phx.set_config(v, None)
    assert phx.get_config(phx.VARIANT_SGEMM, 8, 4096, 4096) == "SKINNY"
    _check("sgemm", 8, 4096, 4096, 1.0, 0.5, "int3", seed=13)
    _check("f16tc", 8, 4096, 4096, 1.0, 0.5, "int3", seed=13)
