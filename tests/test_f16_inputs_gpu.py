"""Half-precision operands (the matrix-multiplication lab's cuBLAS f16 GEMM, Part 4 and
Part 5) through phx_gemm_f16in_f32acc and phx_gemm_f16in_f16out on a GB300.

A and B are f16 already, so the products are the same f16 x f16 products as in the rounding
variant and the oracle is the same float64 sum (its f16 rounding of the inputs is the
identity here).  With an f32 result each element must lie within
8 * sqrt(K) * 2^-24 * (|alpha| sum|a||b| + |beta||C|) of the oracle, bit for bit on integer
inputs.  With an f16 result the oracle rounds float64 straight to f16 once; the kernel
rounds its f32 epilogue value to f16, so the two may differ by the f32 bound plus one f16
unit in the last place, and are bit-identical on integer inputs (whose f32 values are exact).
"""
import itertools

import numpy as np
import pytest

import oracle
from dense_gemm_04_gb300 import phx, synth
from tests.gpu_util import assert_bits_equal, assert_within_bound, bound

pytestmark = pytest.mark.gpu

OPS = list(itertools.product((phx.OP_N, phx.OP_T), repeat=2))


@pytest.fixture(autouse=True)
def _status():
    phx.set_config(phx.VARIANT_F16TC, None)
    yield
    phx.set_config(phx.VARIANT_F16TC, None)
    assert phx.check_device_status() == phx.PHX_OK


def _stored(X, op):
    return np.ascontiguousarray(X.T if op == phx.OP_T else X)


def _run(A, B, C, alpha, beta, out_f16, op_a=phx.OP_N, op_b=phx.OP_N, offset=0):
    """The entry point on device copies: A, B as f16 (stored per op), C as f32 or f16.
    `offset` halves of padding in front of A and B leave them only 2-byte aligned."""
    import torch
    M, K = A.shape
    N = B.shape[1]

    def dev16(x):
        flat = torch.zeros(x.size + offset, dtype=torch.float16)
        flat[offset:] = torch.from_numpy(x.reshape(-1).astype(np.float16))
        return flat.cuda()

    dA, dB = dev16(_stored(A, op_a)), dev16(_stored(B, op_b))
    dC = torch.from_numpy(C.astype(np.float16) if out_f16 else C.copy()).cuda()
    fn = phx.phx_gemm_f16in_f16out if out_f16 else phx.phx_gemm_f16in_f32acc
    st = fn(op_a, op_b, M, N, K, alpha, dA.data_ptr() + 2 * offset, dB.data_ptr() + 2 * offset, beta,
            dC.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    got = dC.cpu().numpy()
    return st, (got.view(np.uint16) if out_f16 else got)


def _f16_ulp(bits):
    """One unit in the last place of each f16 value (2^-24 for subnormals and zero)."""
    e = ((bits.astype(np.int32) >> 10) & 0x1F)
    return np.ldexp(1.0, np.maximum(e, 1) - 25)


def _check(M, N, K, alpha, beta, dist, out_f16, seed=0, op_a=phx.OP_N, op_b=phx.OP_N, offset=0):
    A, B, C = synth.problem(M, N, K, seed=seed, dist=dist)
    if out_f16:
        C = C.astype(np.float16).astype(np.float32)   # an f16 C holds f16 values
    st, got = _run(A, B, C, alpha, beta, out_f16, op_a, op_b, offset)
    assert st == phx.PHX_OK, phx.status_string(st)
    what = f"f16 in, {'f16' if out_f16 else 'f32'} out {(M, N, K)} {dist} ops=({op_a},{op_b}) " \
           f"[{phx.get_config(phx.VARIANT_F16TC, M, N, K)}]"
    if not out_f16:
        want, mag = oracle.gemm(A, B, C, alpha, beta)
        if dist == "int3":
            assert_bits_equal(got, want, what)
        else:
            assert_within_bound(got, want, mag, C, K, alpha, beta, what)
        return
    want, mag = oracle.gemm_f16out(A, B, C, alpha, beta)
    if dist == "int3" and float(alpha).is_integer() and float(2 * beta).is_integer():
        assert np.array_equal(got, want), what
        return
    g = got.view(np.float16).astype(np.float64)
    w = want.view(np.float16).astype(np.float64)
    tol = bound(mag, C, K, alpha, beta) + np.maximum(_f16_ulp(got), _f16_ulp(want))
    bad = ~(np.abs(g - w) <= tol)
    assert not bad.any(), (what, int(bad.sum()), np.argwhere(bad)[:3].tolist())


@pytest.mark.parametrize("out_f16", [False, True])
@pytest.mark.parametrize("shape", [(256, 256, 256), (301, 263, 197), (129, 65, 64), (5, 3, 7), (1, 1, 1),
                                   (1000, 900, 700), (64, 4096, 4096)])
def test_f16_inputs_parity(shape, out_f16):
    M, N, K = shape
    _check(M, N, K, 1.5, 0.5, "int3", out_f16, seed=1)
    _check(M, N, K, 2.0, -1.0, "f16grid", out_f16, seed=2)


@pytest.mark.parametrize("out_f16", [False, True])
def test_f16_inputs_every_config(out_f16):
    # every tile configuration (the skinny one maps to the default tile)
    for name in phx.config_names(phx.VARIANT_F16TC):
        phx.set_config(phx.VARIANT_F16TC, name)
        _check(301, 263, 197, 2.0, -1.0, "int3", out_f16, seed=3)
        _check(256, 256, 256, 1.5, 0.5, "f16grid", out_f16, seed=4)


@pytest.mark.parametrize("out_f16", [False, True])
def test_f16_inputs_split_k(out_f16):
    # a grid too small for the GPU is split along K; an f16 result is rounded once at the end
    _check(1024, 1024, 16384, 2.0, -1.0, "int3", out_f16, seed=5)
    _check(256, 512, 8192, 1.0, 0.5, "f16grid", out_f16, seed=6)


@pytest.mark.parametrize("out_f16", [False, True])
def test_f16_inputs_layouts_and_alignment(out_f16):
    for op_a, op_b in OPS:
        _check(200, 136, 72, 1.0, 0.5, "int3", out_f16, seed=7, op_a=op_a, op_b=op_b)
        _check(130, 70, 100, 1.0, 0.5, "f16grid", out_f16, seed=8, op_a=op_a, op_b=op_b)
    # operands only 2-byte aligned (A is copied instead of read in place); K not a multiple of 8
    _check(200, 136, 72, 1.0, 0.5, "int3", out_f16, seed=9, offset=1)
    _check(200, 136, 77, 1.0, 0.5, "int3", out_f16, seed=10)


@pytest.mark.parametrize("N,c_offset", [(264, 0), (264, 1), (262, 0)])
def test_f16_output_epilogues(N, c_offset):
    # an f16 C with N % 8 == 0 on 16 bytes leaves through the TMA epilogue (c_old loaded a chunk
    # ahead); one 2 bytes off, or with N % 8 != 0, through the register epilogue: the same bits
    import torch
    M, K = 300, 200
    A, B, C = synth.problem(M, N, K, seed=12, dist="int3")
    C = C.astype(np.float16).astype(np.float32)
    want, _ = oracle.gemm_f16out(A, B, C, 1.5, 0.5)
    flat = torch.zeros(M * N + c_offset, dtype=torch.float16)
    flat[c_offset:] = torch.from_numpy(C.reshape(-1).astype(np.float16))
    dC = flat.cuda()
    dA = torch.from_numpy(A.astype(np.float16)).cuda()
    dB = torch.from_numpy(B.astype(np.float16)).cuda()
    st = phx.phx_gemm_f16in_f16out(phx.OP_N, phx.OP_N, M, N, K, 1.5, dA.data_ptr(), dB.data_ptr(), 0.5,
                                   dC.data_ptr() + 2 * c_offset, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == phx.PHX_OK, phx.status_string(st)
    got = dC.cpu()[c_offset:].numpy().view(np.uint16).reshape(M, N)
    assert np.array_equal(got, want), (N, c_offset, int((got != want).sum()))


@pytest.mark.parametrize("out_f16", [False, True])
def test_f16_inputs_degenerate(out_f16):
    A, B, C = synth.problem(9, 7, 5, seed=11, dist="int3")
    # alpha == 0: C <- beta * C
    st, got = _run(A, B, C, 0.0, 0.5, out_f16)
    assert st == phx.PHX_OK
    want = (0.5 * C.astype(np.float64))
    if out_f16:
        assert np.array_equal(got, want.astype(np.float16).view(np.uint16))
    else:
        assert np.array_equal(got, want.astype(np.float32))
    # beta == 0 with NaN in C: C is not read
    st, got = _run(A, B, np.full_like(C, np.nan), 1.0, 0.0, out_f16)
    assert st == phx.PHX_OK
    vals = got.view(np.float16) if out_f16 else got
    assert np.isfinite(vals.astype(np.float32)).all()


def test_f16_output_overflow_and_rounding():
    # results beyond the f16 range become infinity; exact ties round to even
    M, N, K = 2, 8, 16
    A = np.full((M, K), 64.0, np.float32)
    B = np.full((K, N), 64.0, np.float32)                 # 16 * 4096 = 65536 -> inf
    st, got = _run(A, B, np.zeros((M, N), np.float32), 1.0, 0.0, True)
    assert st == phx.PHX_OK and (got == 0x7C00).all()
    A = np.zeros((1, 8), np.float32)
    A[0, 0] = 2049.0 / 2048.0                             # exact in f16? no: 11 bits -> 1 + 2^-11 rounds
    A = A.astype(np.float16).astype(np.float32)
    B = np.zeros((8, 1), np.float32)
    B[0, 0] = 2049.0                                      # exact integer in f16? 2049 -> 2048 (even)
    B = B.astype(np.float16).astype(np.float32)
    st, got = _run(A, B, np.zeros((1, 1), np.float32), 1.0, 0.0, True)
    want, _ = oracle.gemm_f16out(A, B, np.zeros((1, 1), np.float32), 1.0, 0.0)
    assert st == phx.PHX_OK and np.array_equal(got, want)


def test_binding_gemm_f16():
    import torch
    A, B, C = synth.problem(96, 80, 48, seed=12, dist="int3")
    want32, _ = oracle.gemm(A, B, C, 1.0, 1.0)
    want16, _ = oracle.gemm_f16out(A, B, C, 1.0, 1.0)
    dA = torch.from_numpy(A).cuda().half()
    dBt = torch.from_numpy(np.ascontiguousarray(B.T)).cuda().half()   # stored N x K
    c32 = torch.from_numpy(C.copy()).cuda()
    phx.gemm_f16(dA, dBt.t(), c32, 1.0, 1.0)
    assert_bits_equal(c32.cpu().numpy(), want32, "f32 out")
    c16 = torch.from_numpy(C.copy()).cuda().half()
    phx.gemm_f16(dA, dBt.t(), c16, 1.0, 1.0)
    assert np.array_equal(c16.cpu().numpy().view(np.uint16), want16)
