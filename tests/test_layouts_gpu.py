"""Operands stored transposed (the matrix-multiplication lab's layout sweep, Part 5: the same
products with A, B or both stored transposed), through phx_sgemm_ex and
phx_gemm_f16tc_f32acc_ex on a GB300.

Each case is checked twice: against the oracle on op(A), op(B) (bit for bit on integer
inputs, within 8 * sqrt(K) * 2^-24 * (|alpha| sum|a||b| + |beta||C|) otherwise), and bit for bit
against the plain-layout call on contiguous copies of op(A), op(B): on the tile paths a
transposed operand only changes how the operands are read, not which products are summed in
which order.  (The skinny path's kernel for B stored transposed sums in its own order and
is checked against the oracle only.)
"""
import itertools

import numpy as np
import pytest

import oracle
from dense_gemm_04_gb300 import phx, synth
from tests.gpu_util import VARIANTS, assert_bits_equal, assert_within_bound

pytestmark = pytest.mark.gpu

OPS = list(itertools.product((phx.OP_N, phx.OP_T), repeat=2))
EX = {phx.VARIANT_SGEMM: "phx_sgemm_ex", phx.VARIANT_F16TC: "phx_gemm_f16tc_f32acc_ex"}
PLAIN = {phx.VARIANT_SGEMM: "phx_sgemm", phx.VARIANT_F16TC: "phx_gemm_f16tc_f32acc"}


@pytest.fixture(autouse=True)
def _status():
    yield
    assert phx.check_device_status() == phx.PHX_OK


def _stored(X, op):
    """The array as the caller stores it: X itself for OP_N, its transpose for OP_T."""
    return np.ascontiguousarray(X.T if op == phx.OP_T else X)


def _run_ex(variant, op_a, op_b, A, B, C, alpha, beta, offset=0):
    """phx_*_ex on device copies of op(A) and op(B) stored as op_a / op_b says; `offset`
    floats of padding in front of each operand make its pointer only 4-byte aligned."""
    import torch
    M, K = A.shape
    N = B.shape[1]

    def dev(x):
        flat = torch.zeros(x.size + offset, dtype=torch.float32)
        flat[offset:] = torch.from_numpy(x.reshape(-1))
        return flat.cuda()

    dA, dB = dev(_stored(A, op_a)), dev(_stored(B, op_b))
    dC = torch.from_numpy(np.ascontiguousarray(C)).cuda()
    h = torch.cuda.current_stream().cuda_stream
    st = getattr(phx, EX[variant])(op_a, op_b, M, N, K, alpha, dA.data_ptr() + 4 * offset,
                                   dB.data_ptr() + 4 * offset, beta, dC.data_ptr(), h)
    torch.cuda.synchronize()
    return st, dC.cpu().numpy()


def _run_plain(variant, A, B, C, alpha, beta):
    import torch
    M, K = A.shape
    N = B.shape[1]
    dA, dB, dC = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (A, B, C))
    st = getattr(phx, PLAIN[variant])(M, N, K, alpha, dA.data_ptr(), dB.data_ptr(), beta, dC.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == phx.PHX_OK, phx.status_string(st)
    return dC.cpu().numpy()


# shapes: aligned; ragged in every direction across several 64-wide transpose tiles; odd
# extents (no 16-byte rows, so the transposing pass takes its scalar loads); K below one
# k block; a degenerate vector
SHAPES = [(256, 256, 256), (301, 263, 197), (129, 65, 63), (67, 131, 4093), (5, 3, 7), (1, 1, 1),
          (1, 200, 9)]


@pytest.mark.parametrize("vname", list(VARIANTS))
@pytest.mark.parametrize("op_a,op_b", OPS)
@pytest.mark.parametrize("shape", SHAPES)
def test_layout_parity(vname, op_a, op_b, shape):
    variant, f16 = VARIANTS[vname]
    M, N, K = shape
    for dist, seed in (("int3", 1), ("uniform", 2)):
        A, B, C = synth.problem(M, N, K, seed=seed, dist=dist)
        alpha, beta = 2.0, -1.0
        st, got = _run_ex(variant, op_a, op_b, A, B, C, alpha, beta)
        assert st == phx.PHX_OK, phx.status_string(st)
        what = f"{vname} ops=({op_a},{op_b}) {shape} {dist}"
        want, mag = oracle.gemm(A, B, C, alpha, beta, f16_inputs=f16)
        if dist == "int3":
            assert_bits_equal(got, want, what)
        else:
            assert_within_bound(got, want, mag, C, K, alpha, beta, what)
        # the tile paths copy (or round) a transposed operand into the plain layout and run the
        # same kernels; the skinny path has a kernel of its own for B stored transposed, which
        # sums in another order (the oracle check above covers it)
        if not (op_b == phx.OP_T and phx.get_config(variant, M, N, K) == "SKINNY"):
            assert_bits_equal(got, _run_plain(variant, A, B, C, alpha, beta), what + " vs plain layout")


@pytest.mark.parametrize("vname", list(VARIANTS))
def test_layout_unaligned_pointers(vname):
    # operands that start 4 bytes past a 16-byte boundary take the scalar loads
    variant, f16 = VARIANTS[vname]
    M, N, K = 200, 136, 72
    A, B, C = synth.problem(M, N, K, seed=4, dist="int3")
    want, _ = oracle.gemm(A, B, C, 1.0, 0.5, f16_inputs=f16)
    for op_a, op_b in OPS:
        st, got = _run_ex(variant, op_a, op_b, A, B, C, 1.0, 0.5, offset=1)
        assert st == phx.PHX_OK, phx.status_string(st)
        assert_bits_equal(got, want, f"{vname} ops=({op_a},{op_b}) unaligned")


@pytest.mark.parametrize("vname", list(VARIANTS))
def test_layout_degenerate(vname):
    variant, _ = VARIANTS[vname]
    A, B, C = synth.problem(9, 7, 5, seed=5, dist="int3")
    for op_a, op_b in OPS:
        # alpha == 0: A and B are not read, C <- beta * C
        st, got = _run_ex(variant, op_a, op_b, A, B, C, 0.0, 2.0)
        assert st == phx.PHX_OK
        assert_bits_equal(got, (2.0 * C).astype(np.float32), "alpha = 0")
        # beta == 0 with NaN in C: C is not read
        Cn = np.full_like(C, np.nan)
        st, got = _run_ex(variant, op_a, op_b, A, B, Cn, 1.0, 0.0)
        assert st == phx.PHX_OK and np.isfinite(got).all()


@pytest.mark.parametrize("vname", list(VARIANTS))
def test_layout_full_size_matches_plain(vname):
    # 4096^3 in every storage order: bit-identical to the plain layout on the same values
    import torch
    variant, _ = VARIANTS[vname]
    n = 4096
    g = torch.Generator(device="cuda").manual_seed(0)
    A = torch.rand(n, n, device="cuda", generator=g) * 2 - 1
    B = torch.rand(n, n, device="cuda", generator=g) * 2 - 1
    C0 = torch.rand(n, n, device="cuda", generator=g) * 2 - 1
    At, Bt = A.t().contiguous(), B.t().contiguous()
    h = torch.cuda.current_stream().cuda_stream
    ref = C0.clone()
    phx.check(getattr(phx, PLAIN[variant])(n, n, n, 1.0, A.data_ptr(), B.data_ptr(), 0.5, ref.data_ptr(), h))
    for op_a, op_b in OPS:
        C = C0.clone()
        a = At if op_a == phx.OP_T else A
        b = Bt if op_b == phx.OP_T else B
        phx.check(getattr(phx, EX[variant])(op_a, op_b, n, n, n, 1.0, a.data_ptr(), b.data_ptr(), 0.5,
                                            C.data_ptr(), h))
        torch.cuda.synchronize()
        assert torch.equal(C, ref), (vname, op_a, op_b)


def test_binding_takes_transpose_views():
    import torch
    A, B, C = synth.problem(96, 80, 48, seed=6, dist="int3")
    want, _ = oracle.gemm(A, B, C, 1.0, 1.0, f16_inputs=False)
    dAt = torch.from_numpy(np.ascontiguousarray(A.T)).cuda()   # stored K x M
    dBt = torch.from_numpy(np.ascontiguousarray(B.T)).cuda()   # stored N x K
    for fn in (phx.sgemm, phx.gemm_f16tc_f32acc):
        dC = torch.from_numpy(C.copy()).cuda()
        fn(dAt.t(), dBt.t(), dC, 1.0, 1.0)
        assert_bits_equal(dC.cpu().numpy(), want, fn.__name__)
