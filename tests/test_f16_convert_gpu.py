"""The f16 tensor-core GEMM whose kernel rounds A or B itself (the CONVERT_A=1 and
CONVERT_B=1 configurations), through the C ABI on a GB300.

Its converter warps write the rounded halves into the 128-byte swizzled shared-memory layout
that the TMA path writes (B transposed on the way, one n per row), so the tensor cores see
the same operands: on integer-valued inputs it must match the oracle bit for bit, on uniform
inputs stay within the bound, and where the other kernel runs the same MMA sequence (one CTA
per 128 x TILE_N tile, one whole wave, no split along K) the two must agree bit for bit on
any inputs.  A mistake in the layout (a swizzle, a row, a column or a chunk out of place)
would show in every one of these.
"""
import numpy as np
import pytest

import oracle
from dense_gemm_04_gb300 import phx, synth
from tests.gpu_util import assert_bits_equal, assert_within_bound

pytestmark = pytest.mark.gpu

_NAMES = phx.config_names(phx.VARIANT_F16TC)
CVT = [n for n in _NAMES if "CONVERT_A=1" in n and "CONVERT_B=1" not in n]      # A rounded here
CVTB = [n for n in _NAMES if "CONVERT_B=1" in n and "CONVERT_A=1" not in n]     # B rounded here
CVTAB = [n for n in _NAMES if "CONVERT_A=1" in n and "CONVERT_B=1" in n]        # both


@pytest.fixture(autouse=True)
def _unpin():
    phx.set_config(phx.VARIANT_F16TC, None)
    yield
    phx.set_config(phx.VARIANT_F16TC, None)
    assert phx.check_device_status() == phx.PHX_OK


def _run(A, B, C, alpha, beta, a_offset=0, op_a=phx.OP_N, op_b=phx.OP_N, b_offset=0):
    """The f16 call on device copies; A (B) starts a_offset (b_offset) floats into its buffer.
    With op_a or op_b = OP_T the operand is passed in its transposed storage (A.T or B.T
    contiguous)."""
    import torch
    M, K = A.shape
    N = B.shape[1]

    def dev(x, offset):
        buf = torch.zeros(x.size + offset, dtype=torch.float32, device="cuda")
        buf[offset:] = torch.from_numpy(x.ravel()).cuda()
        return buf, buf.data_ptr() + 4 * offset

    abuf, a_ptr = dev(np.ascontiguousarray(A.T if op_a == phx.OP_T else A), a_offset)
    bbuf, b_ptr = dev(np.ascontiguousarray(B.T if op_b == phx.OP_T else B), b_offset)
    dC = torch.from_numpy(np.ascontiguousarray(C)).cuda()
    s = torch.cuda.current_stream().cuda_stream
    if op_a == phx.OP_N and op_b == phx.OP_N:
        st = phx.phx_gemm_f16tc_f32acc(M, N, K, alpha, a_ptr, b_ptr, beta, dC.data_ptr(), s)
    else:
        st = phx.phx_gemm_f16tc_f32acc_ex(op_a, op_b, M, N, K, alpha, a_ptr, b_ptr, beta, dC.data_ptr(), s)
    torch.cuda.synchronize()
    return st, dC.cpu().numpy()


SHAPES = [
    (300, 100, 700, 1.5, 0.5),     # ragged in every dimension
    (257, 64, 130, 1.0, -1.0),     # K % 4 != 0: A rows not on 16 bytes, 4-byte loads
    (1000, 300, 1000, 2.0, 0.0),   # N > TILE_N: several tile columns; beta = 0 (C not read)
    (128, 256, 64, 1.0, 0.5),      # one tile, one k block
    (5, 7, 3, 1.0, 0.5),           # smaller than a tile in every dimension
    (20000, 96, 520, 1.0, 0.5),    # more tiles than SMs: the persistent loop, and a k tail
    (1030, 130, 4100, 1.0, 0.5),   # long K with a tail; N % 4 != 0 (the 4-byte epilogue)
]


SHAPES_B = [
    (64, 4096, 4096, 1.0, 0.5),    # few rows: K split into slices of partial planes, then reduced
    (17, 3000, 700, 1.5, 0.5),     # ragged; N % 4 != 0: B's rows not on 16 bytes, 4-byte loads
    (200, 1500, 1030, 2.0, -1.0),  # two tile rows; a k tail
    (128, 256, 64, 1.0, 0.0),      # one tile, one k block, beta = 0
    (5, 7, 3, 1.0, 0.5),           # smaller than a tile in every dimension
    (300, 100, 700, 1.5, 0.5),     # more rows than two tiles
]


SHAPES_AB = [
    (300, 200, 700, 1.5, 0.5),     # ragged in every dimension
    (256, 256, 4096, 1.0, 0.5),    # 4 tiles: K split into 8 slices of partial planes
    (257, 130, 130, 2.0, -1.0),    # K % 4 != 0: A's rows not on 16 bytes; N % 4 != 0
    (5, 7, 3, 1.0, 0.5),           # smaller than a tile in every dimension
    (1024, 1024, 1024, 1.0, 0.0),  # a whole wave of tiles, beta = 0
]


@pytest.mark.parametrize("cfg", CVT + CVTB + CVTAB)
@pytest.mark.parametrize("dist", ["int3", "uniform"])
def test_matches_the_oracle(cfg, dist):
    phx.set_config(phx.VARIANT_F16TC, cfg)
    shapes = SHAPES if cfg in CVT else SHAPES_B if cfg in CVTB else SHAPES_AB
    for i, (M, N, K, alpha, beta) in enumerate(shapes):
        A, B, C = synth.problem(M, N, K, seed=40 + i, dist=dist)
        want, mag = oracle.gemm(A, B, C, alpha, beta, f16_inputs=True)
        st, got = _run(A, B, C, alpha, beta)
        assert st == phx.PHX_OK, phx.status_string(st)
        assert phx.last_config(phx.VARIANT_F16TC) == cfg
        what = f"[{cfg}] {(M, N, K)} {dist}"
        if dist == "int3":
            assert_bits_equal(got, want, what)
        else:
            assert_within_bound(got, want, mag, C, K, alpha, beta, what)


@pytest.mark.parametrize("cfg", CVT)
def test_unaligned_a_and_transposed_b(cfg):
    # A one float past a 16-byte boundary: the converters load 4 bytes at a time
    phx.set_config(phx.VARIANT_F16TC, cfg)
    M, N, K = 700, 200, 516
    A, B, C = synth.problem(M, N, K, seed=7, dist="int3")
    want, _ = oracle.gemm(A, B, C, 1.0, 0.5, f16_inputs=True)
    st, got = _run(A, B, C, 1.0, 0.5, a_offset=1)
    assert st == phx.PHX_OK
    assert_bits_equal(got, want, f"[{cfg}] A unaligned")
    # B stored N x K: the rounding pass reads it in that order
    st, got = _run(A, B, C, 1.0, 0.5, op_b=phx.OP_T)
    assert st == phx.PHX_OK
    assert_bits_equal(got, want, f"[{cfg}] B transposed")
    # A stored K x M: this kernel reads A as M x K only, so the call takes the other kernel
    st, got = _run(A, B, C, 1.0, 0.5, op_a=phx.OP_T)
    assert st == phx.PHX_OK
    assert "CONVERT_A" not in phx.last_config(phx.VARIANT_F16TC)
    assert_bits_equal(got, want, f"[{cfg}] A transposed")


@pytest.mark.parametrize("cfg", CVTB)
def test_unaligned_b_and_transposed_operands(cfg):
    # B one float past a 16-byte boundary: the converters load it 4 bytes at a time
    phx.set_config(phx.VARIANT_F16TC, cfg)
    M, N, K = 100, 1200, 516
    A, B, C = synth.problem(M, N, K, seed=8, dist="int3")
    want, _ = oracle.gemm(A, B, C, 1.0, 0.5, f16_inputs=True)
    st, got = _run(A, B, C, 1.0, 0.5, b_offset=1)
    assert st == phx.PHX_OK
    assert_bits_equal(got, want, f"[{cfg}] B unaligned")
    # A stored K x M: the rounding pass reads it in that order
    st, got = _run(A, B, C, 1.0, 0.5, op_a=phx.OP_T)
    assert st == phx.PHX_OK
    assert_bits_equal(got, want, f"[{cfg}] A transposed")
    # B stored N x K: this kernel reads B as K x N only, so the call takes the other kernel
    st, got = _run(A, B, C, 1.0, 0.5, op_b=phx.OP_T)
    assert st == phx.PHX_OK
    assert "CONVERT" not in phx.last_config(phx.VARIANT_F16TC)
    assert_bits_equal(got, want, f"[{cfg}] B transposed")


@pytest.mark.parametrize("tile_n,stages", [(64, 8), (128, 6), (256, 4)])
def test_same_bits_as_the_tma_kernel(tile_n, stages):
    # 152 tiles of 128 x TILE_N on 152 SMs: the other kernel runs one whole wave of whole
    # tiles (no half-width tail items, no split along K), the same MMA sequence per tile
    import torch
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the single-wave shape is sized for 152 SMs")
    M, N, K = 152 * 128, tile_n, 512
    A, B, C = synth.problem(M, N, K, seed=3, dist="uniform")
    base = f"TILE_M=128 TILE_N={tile_n} TILE_K=64 STAGES={stages}"
    phx.set_config(phx.VARIANT_F16TC, base)
    st, tma = _run(A, B, C, 1.25, -0.5)
    assert st == phx.PHX_OK and phx.last_config(phx.VARIANT_F16TC) == base
    phx.set_config(phx.VARIANT_F16TC, f"TILE_M=128 TILE_N={tile_n} TILE_K=64 CONVERT_A=1")
    st, cvt = _run(A, B, C, 1.25, -0.5)
    assert st == phx.PHX_OK and "CONVERT_A=1" in phx.last_config(phx.VARIANT_F16TC)
    assert_bits_equal(cvt, tma, f"TILE_N={tile_n}: A rounded in the kernel vs by the pass")


@pytest.mark.parametrize("tile_n,stages", [(64, 8), (128, 6)])
def test_b_rounded_in_the_kernel_same_bits_as_the_tma_kernel(tile_n, stages):
    # one row of 152 tiles of 128 x TILE_N on 152 SMs, K short enough not to split
    import torch
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the single-wave shape is sized for 152 SMs")
    M, N, K = 128, 152 * tile_n, 512
    A, B, C = synth.problem(M, N, K, seed=4, dist="uniform")
    base = f"TILE_M=128 TILE_N={tile_n} TILE_K=64 STAGES={stages}"
    phx.set_config(phx.VARIANT_F16TC, base)
    st, tma = _run(A, B, C, 1.25, -0.5)
    assert st == phx.PHX_OK and phx.last_config(phx.VARIANT_F16TC) == base
    phx.set_config(phx.VARIANT_F16TC, f"TILE_M=128 TILE_N={tile_n} TILE_K=64 CONVERT_B=1")
    st, cvt = _run(A, B, C, 1.25, -0.5)
    assert st == phx.PHX_OK and "CONVERT_B=1" in phx.last_config(phx.VARIANT_F16TC)
    assert_bits_equal(cvt, tma, f"TILE_N={tile_n}: B rounded in the kernel vs by the pass")


@pytest.mark.parametrize("cfg", CVTAB)
def test_both_rounded_unaligned_and_transposed(cfg):
    phx.set_config(phx.VARIANT_F16TC, cfg)
    M, N, K = 300, 264, 516
    A, B, C = synth.problem(M, N, K, seed=9, dist="int3")
    want, _ = oracle.gemm(A, B, C, 1.0, 0.5, f16_inputs=True)
    # either operand off 16 bytes: no tensor maps, the converters load both themselves
    for a_off, b_off in ((1, 0), (0, 1)):
        st, got = _run(A, B, C, 1.0, 0.5, a_offset=a_off, b_offset=b_off)
        assert st == phx.PHX_OK
        assert phx.last_config(phx.VARIANT_F16TC) == cfg
        assert_bits_equal(got, want, f"[{cfg}] offsets {a_off}, {b_off}")
    # an operand stored transposed takes the kernels without this one
    for op_a, op_b in ((phx.OP_T, phx.OP_N), (phx.OP_N, phx.OP_T)):
        st, got = _run(A, B, C, 1.0, 0.5, op_a=op_a, op_b=op_b)
        assert st == phx.PHX_OK
        assert "CONVERT" not in phx.last_config(phx.VARIANT_F16TC)
        assert_bits_equal(got, want, f"[{cfg}] ops {op_a}, {op_b}")


@pytest.mark.parametrize("tile_n,stages", [(64, 8), (128, 6)])
def test_both_rounded_same_bits_as_the_tma_kernel(tile_n, stages):
    # 152 tiles of 128 x TILE_N, one whole wave, K short enough not to split
    import torch
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the single-wave shape is sized for 152 SMs")
    M, N, K = 8 * 128, 19 * tile_n, 512
    A, B, C = synth.problem(M, N, K, seed=6, dist="uniform")
    base = f"TILE_M=128 TILE_N={tile_n} TILE_K=64 STAGES={stages}"
    phx.set_config(phx.VARIANT_F16TC, base)
    st, tma = _run(A, B, C, 1.25, -0.5)
    assert st == phx.PHX_OK and phx.last_config(phx.VARIANT_F16TC) == base
    phx.set_config(phx.VARIANT_F16TC, f"TILE_M=128 TILE_N={tile_n} TILE_K=64 CONVERT_A=1 CONVERT_B=1")
    st, cvt = _run(A, B, C, 1.25, -0.5)
    assert st == phx.PHX_OK and "CONVERT_A=1 CONVERT_B=1" in phx.last_config(phx.VARIANT_F16TC)
    assert_bits_equal(cvt, tma, f"TILE_N={tile_n}: both rounded in the kernel vs by the pass")


def test_default_routes_few_rows_here():
    # (64, 4096, 4096): B is 64 MiB of f32 against 1 MiB of A; K split into planes
    M, N, K = 64, 4096, 4096
    assert "CONVERT_B=1" in phx.get_config(phx.VARIANT_F16TC, M, N, K)
    assert phx.get_config(phx.VARIANT_F16TC, 8, N, K) == "SKINNY"
    assert "CONVERT_B=1" in phx.get_config(phx.VARIANT_F16TC, 12, N, K)
    A, B, C = synth.problem(M, N, K, seed=13, dist="int3")
    want, _ = oracle.gemm(A, B, C, 1.0, 0.5, f16_inputs=True)
    st, got = _run(A, B, C, 1.0, 0.5)
    assert st == phx.PHX_OK
    assert "CONVERT_B=1" in phx.last_config(phx.VARIANT_F16TC)
    assert_bits_equal(got, want, "(64, 4096, 4096)")


def test_default_routes_tall_narrow_problems_here():
    # (16384, 128, 4096): A is 256 MiB of f32 against 2 MiB of B; checked on sampled rows
    M, N, K = 16384, 128, 4096
    assert "CONVERT_A=1" in phx.get_config(phx.VARIANT_F16TC, M, N, K)
    assert "CONVERT_A" not in phx.get_config(phx.VARIANT_F16TC, 4096, 4096, 4096)
    A, B, C = synth.problem(M, N, K, seed=11, dist="int3")
    st, got = _run(A, B, C, 1.0, 0.5)
    assert st == phx.PHX_OK
    assert "CONVERT_A=1" in phx.last_config(phx.VARIANT_F16TC)
    rows = np.random.default_rng(0).choice(M, 512, replace=False)
    rows.sort()
    want, _ = oracle.gemm(A[rows], B, C[rows], 1.0, 0.5, f16_inputs=True)
    assert_bits_equal(got[rows], want, "(16384, 128, 4096) sampled rows")


def test_default_routes_fewer_rows_split_k_here():
    # (2085, 96, 4100): 17 row tiles, too few for the SMs; the kernel that rounds A splits K
    # (65 k blocks: 8 slices of 9, the last of 2) into partial planes.  Whole result, bit for
    # bit on integers.
    M, N, K = 2085, 96, 4100
    assert phx.get_config(phx.VARIANT_F16TC, M, N, K).endswith(" CONVERT_A=1")
    A, B, C = synth.problem(M, N, K, seed=17, dist="int3")
    want, _ = oracle.gemm(A, B, C, 2.0, -1.0, f16_inputs=True)
    st, got = _run(A, B, C, 2.0, -1.0)
    assert st == phx.PHX_OK
    assert phx.last_config(phx.VARIANT_F16TC).endswith(" CONVERT_A=1")
    assert_bits_equal(got, want, "(2085, 96, 4100)")


def test_f16_operand_entry_points_take_the_tma_kernel():
    # phx_gemm_f16in_* read f16 operands: a CONVERT pin gives way to the default tile there
    import torch
    phx.set_config(phx.VARIANT_F16TC, CVT[1])
    M, N, K = 300, 128, 256
    A, B, C = synth.problem(M, N, K, seed=5, dist="int3")
    want, _ = oracle.gemm(A, B, C, 1.0, 0.0, f16_inputs=True)
    dA = torch.from_numpy(A).cuda().half()
    dB = torch.from_numpy(B).cuda().half()
    dC = torch.zeros(M, N, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = phx.phx_gemm_f16in_f32acc(phx.OP_N, phx.OP_N, M, N, K, 1.0, dA.data_ptr(), dB.data_ptr(), 0.0,
                                   dC.data_ptr(), s)
    torch.cuda.synchronize()
    assert st == phx.PHX_OK
    assert "CONVERT_A" not in phx.last_config(phx.VARIANT_F16TC)
    assert_bits_equal(dC.cpu().numpy(), want, "f16 operands with a CONVERT_A pin")
