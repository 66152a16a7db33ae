"""Parity of the CUDA path with the oracle, through the C ABI, on a GB300.

Integer-valued inputs make every partial sum exact in f32, so on them both precisions must
match the oracle bit for bit.  On uniform [-1, 1) inputs each element must lie within
8 * sqrt(K) * 2^-24 * (|alpha| * sum_k |a_ik||b_kj| + |beta| * |C_ij|) of the oracle.
"""
import numpy as np
import pytest

import oracle
from dense_gemm_04_gb300 import phx, synth
from tests.gpu_util import VARIANTS, assert_bits_equal, assert_within_bound, run_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _unpin():
    phx.set_config(phx.VARIANT_SGEMM, None)
    phx.set_config(phx.VARIANT_F16TC, None)
    yield
    phx.set_config(phx.VARIANT_SGEMM, None)
    phx.set_config(phx.VARIANT_F16TC, None)
    assert phx.check_device_status() == phx.PHX_OK


def _check(variant_name, M, N, K, alpha, beta, dist, seed=0, exact=None):
    variant, f16 = VARIANTS[variant_name]
    A, B, C = synth.problem(M, N, K, seed=seed, dist=dist)
    want, mag = oracle.gemm(A, B, C, alpha, beta, f16_inputs=f16)
    st, got = run_cuda(variant, A, B, C, alpha, beta)
    assert st == phx.PHX_OK, phx.status_string(st)
    what = f"{variant_name} {(M, N, K)} {dist} a={alpha} b={beta} [{phx.get_config(variant, M, N, K)}]"
    if exact if exact is not None else dist == "int3":
        assert_bits_equal(got, want, what)
    else:
        assert_within_bound(got, want, mag, C, K, alpha, beta, what)


# ----------------------------------------------------------------------------------------
# The 256^3 correctness config, every compiled configuration of both variants
# ----------------------------------------------------------------------------------------

def _all_configs():
    out = []
    for vname, (variant, _) in VARIANTS.items():
        for name in phx.config_names(variant):
            out.append((vname, name))
    return out


@pytest.mark.parametrize("vname,cfg", _all_configs())
def test_every_config_256_cubed(vname, cfg):
    variant, _ = VARIANTS[vname]
    phx.set_config(variant, cfg)
    _check(vname, 256, 256, 256, 1.5, 0.5, "int3")
    _check(vname, 256, 256, 256, 1.5, 0.5, "uniform")


@pytest.mark.parametrize("vname,cfg", _all_configs())
def test_every_config_masked(vname, cfg):
    # every dimension ragged, several tiles and several k blocks in every direction
    variant, _ = VARIANTS[vname]
    phx.set_config(variant, cfg)
    _check(vname, 301, 263, 197, 2.0, -1.0, "int3")
    _check(vname, 301, 263, 197, 2.0, -1.0, "uniform", seed=3)


# ----------------------------------------------------------------------------------------
# Edge sweep: tiny and ragged shapes (default configuration choice)
# ----------------------------------------------------------------------------------------

EDGE_DIMS = [1, 2, 3, 15, 16, 17, 63, 64, 65, 127, 128, 129]


def _edge_shapes():
    rng = np.random.default_rng(7)
    shapes = {(d, d, d) for d in EDGE_DIMS}
    while len(shapes) < 40:
        shapes.add(tuple(int(x) for x in rng.choice(EDGE_DIMS, 3)))
    return sorted(shapes)


@pytest.mark.parametrize("vname", list(VARIANTS))
def test_edge_sweep(vname):
    for M, N, K in _edge_shapes():
        _check(vname, M, N, K, 1.5, 0.5, "int3")
        _check(vname, M, N, K, -0.75, 1.25, "uniform", seed=M * 1000 + N * 10 + K)


@pytest.mark.parametrize("vname", list(VARIANTS))
def test_k_tail_and_long_k(vname):
    # K just around the stage ring and the k-block sizes: every pipeline phase wraps
    for K in (7, 8, 9, 63, 64, 65, 255, 257, 1000, 4100):
        _check(vname, 130, 70, K, 1.0, 0.5, "int3")
        _check(vname, 130, 70, K, 1.0, 0.5, "uniform", seed=K)


@pytest.mark.parametrize("vname", list(VARIANTS))
def test_guard_band_canaries(vname):
    """No write outside C: C sits inside a larger buffer whose margins hold a sentinel."""
    import torch
    variant, f16 = VARIANTS[vname]
    M, N, K = 131, 77, 45
    A, B, C = synth.problem(M, N, K, seed=5, dist="int3")
    want, _ = oracle.gemm(A, B, C, 2.0, -1.0, f16_inputs=f16)
    pad = 4096
    buf = torch.full((pad + M * N + pad,), 12345.0, dtype=torch.float32, device="cuda")
    buf[pad:pad + M * N] = torch.from_numpy(C.reshape(-1)).cuda()
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    fn = phx.phx_sgemm if variant == phx.VARIANT_SGEMM else phx.phx_gemm_f16tc_f32acc
    st = fn(M, N, K, 2.0, dA.data_ptr(), dB.data_ptr(), -1.0, buf.data_ptr() + 4 * pad,
            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == phx.PHX_OK
    h = buf.cpu().numpy()
    assert (h[:pad] == 12345.0).all() and (h[pad + M * N:] == 12345.0).all()
    assert_bits_equal(h[pad:pad + M * N].reshape(M, N), want, vname)


# ----------------------------------------------------------------------------------------
# Degenerate cases of the method
# ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("vname", list(VARIANTS))
def test_beta_zero_does_not_read_c(vname):
    variant, f16 = VARIANTS[vname]
    A, B, _ = synth.problem(70, 90, 33, seed=2, dist="int3")
    C = np.full((70, 90), np.nan, dtype=np.float32)
    want, _ = oracle.gemm(A, B, C, 1.5, 0.0, f16_inputs=f16)
    st, got = run_cuda(variant, A, B, C, 1.5, 0.0)
    assert st == phx.PHX_OK and not np.isnan(got).any()
    assert_bits_equal(got, want, vname)


@pytest.mark.parametrize("vname", list(VARIANTS))
@pytest.mark.parametrize("alpha,K", [(0.0, 40), (1.0, 0), (0.0, 0)])
def test_alpha_zero_or_k_zero_scales_c(vname, alpha, K):
    variant, _ = VARIANTS[vname]
    M, N = 50, 60
    A = np.full((M, K), np.nan, dtype=np.float32)   # must not be read
    B = np.full((K, N), np.nan, dtype=np.float32)
    C = synth.matrix(M, N, seed=1, tensor=2)
    for beta in (0.5, 0.0, 1.0):
        st, got = run_cuda(variant, A, B, C, alpha, beta)
        assert st == phx.PHX_OK
        assert np.array_equal(got, (beta * C.astype(np.float64)).astype(np.float32))


@pytest.mark.parametrize("vname", list(VARIANTS))
def test_empty_and_invalid_calls_touch_nothing(vname):
    import torch
    variant, _ = VARIANTS[vname]
    fn = phx.phx_sgemm if variant == phx.VARIANT_SGEMM else phx.phx_gemm_f16tc_f32acc
    s = torch.cuda.current_stream().cuda_stream
    C = torch.full((8, 8), 7.0, device="cuda")
    A = torch.ones((8, 8), device="cuda")
    assert fn(0, 8, 8, 1.0, A.data_ptr(), A.data_ptr(), 0.0, C.data_ptr(), s) == phx.PHX_OK
    assert fn(8, 0, 8, 1.0, A.data_ptr(), A.data_ptr(), 0.0, C.data_ptr(), s) == phx.PHX_OK
    # C aliasing A is rejected before anything is launched
    assert fn(8, 8, 8, 1.0, C.data_ptr(), A.data_ptr(), 0.0, C.data_ptr(), s) == phx.PHX_ERR_INVALID
    assert fn(8, 8, -1, 1.0, A.data_ptr(), A.data_ptr(), 0.0, C.data_ptr(), s) == phx.PHX_ERR_INVALID
    torch.cuda.synchronize()
    assert (C == 7.0).all()


def test_a_and_b_may_alias():
    import torch
    X = synth.matrix(96, 96, seed=4, dist="int3")
    C = synth.matrix(96, 96, seed=4, tensor=2, dist="int3")
    for vname, (variant, f16) in VARIANTS.items():
        want, _ = oracle.gemm(X, X, C, 1.0, 1.0, f16_inputs=f16)
        dX, dC = torch.from_numpy(X).cuda(), torch.from_numpy(C).cuda()
        fn = phx.phx_sgemm if variant == phx.VARIANT_SGEMM else phx.phx_gemm_f16tc_f32acc
        assert fn(96, 96, 96, 1.0, dX.data_ptr(), dX.data_ptr(), 1.0, dC.data_ptr(),
                  torch.cuda.current_stream().cuda_stream) == phx.PHX_OK
        assert_bits_equal(dC.cpu().numpy(), want, vname)


def test_unaligned_pointers_take_masked_path():
    # 4-byte but not 16-byte aligned operands on a tile-aligned shape
    import torch
    M = N = K = 256
    A, B, C = synth.problem(M, N, K, seed=9, dist="int3")
    for vname, (variant, f16) in VARIANTS.items():
        want, _ = oracle.gemm(A, B, C, 1.5, 0.5, f16_inputs=f16)
        bufs = []
        for x in (A, B, C):
            t = torch.empty(x.size + 1, dtype=torch.float32, device="cuda")
            t[1:] = torch.from_numpy(x.reshape(-1)).cuda()
            bufs.append(t)
        fn = phx.phx_sgemm if variant == phx.VARIANT_SGEMM else phx.phx_gemm_f16tc_f32acc
        st = fn(M, N, K, 1.5, bufs[0].data_ptr() + 4, bufs[1].data_ptr() + 4, 0.5, bufs[2].data_ptr() + 4,
                torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert st == phx.PHX_OK
        assert_bits_equal(bufs[2][1:].cpu().numpy().reshape(M, N), want, vname)


# ----------------------------------------------------------------------------------------
# The lab's error levels (Part 2 ladder, n = 1024, uniform [0, 1), vs float64 of the
# unrounded inputs)
# ----------------------------------------------------------------------------------------

def test_lab_error_levels():
    import os
    rows = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", "lab_error_levels.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                p = line.split()
                rows[p[0]] = (float(p[2]), float(p[3]))
    n = 1024
    A = synth.matrix(n, n, seed=0, tensor=0, dist="unit")
    B = synth.matrix(n, n, seed=0, tensor=1, dist="unit")
    C = np.zeros((n, n), np.float32)
    ref = A.astype(np.float64) @ B.astype(np.float64)

    def errs(out):
        d = out.astype(np.float64) - ref
        return np.abs(d).max() / np.abs(ref).max(), np.linalg.norm(d) / np.linalg.norm(ref)

    st, got32 = run_cuda(phx.VARIANT_SGEMM, A, B, C, 1.0, 0.0)
    e_max, e_fro = errs(got32)
    lab_max, lab_fro = rows["f32"]
    assert st == phx.PHX_OK and e_max <= 2 * lab_max and e_fro <= 2 * lab_fro, (e_max, e_fro)
    st, got16 = run_cuda(phx.VARIANT_F16TC, A, B, C, 1.0, 0.0)
    e_max, e_fro = errs(got16)
    lab_max, lab_fro = rows["f16_in_f32_acc"]
    assert st == phx.PHX_OK
    assert lab_fro / 1.5 <= e_fro <= lab_fro * 1.5 and lab_max / 2 <= e_max <= lab_max * 2, (e_max, e_fro)


# ----------------------------------------------------------------------------------------
# Small grids split along K (the slices' partial products added in slice order) or spread
# as stream-K blocks (f32), and tiles of a last, partial round dealt out as half-width items
# (tensor cores)
# ----------------------------------------------------------------------------------------

TAIL_SHAPES = [(640, 512, 2048), (650, 500, 2000), (5000, 300, 700), (4224, 4096, 256), (129, 257, 4100)]


@pytest.mark.parametrize("vname", list(VARIANTS))
def test_tail_wave_paths(vname):
    variant, _ = VARIANTS[vname]
    for cfg in phx.config_names(variant):
        phx.set_config(variant, cfg)
        for M, N, K in TAIL_SHAPES[:2]:
            _check(vname, M, N, K, 2.0, -1.0, "int3")
            _check(vname, M, N, K, 2.0, -1.0, "uniform", seed=M + K)
    phx.set_config(variant, None)
    for M, N, K in TAIL_SHAPES[2:]:
        _check(vname, M, N, K, 1.5, 0.5, "int3")
        _check(vname, M, N, K, 1.5, 0.5, "uniform", seed=N)


@pytest.mark.parametrize("vname", list(VARIANTS))
def test_results_identical_run_to_run(vname):
    variant, _ = VARIANTS[vname]
    for M, N, K in [(640, 512, 2048), (4096, 4096, 4096)]:
        A, B, C = synth.problem(M, N, K, seed=17)
        outs = [run_cuda(variant, A, B, C, 1.0, 0.5)[1] for _ in range(3)]
        for o in outs[1:]:
            assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32)), (vname, M, N, K)


@pytest.mark.parametrize("shape", [(4096, 4096, 4096), (1000, 1000, 4000), (512, 512, 8192), (4095, 4097, 4093),
                                   (16384, 128, 1024)])
def test_new_inputs_in_reused_workspace(shape):
    # The f16 call's scratch (rounded operand copies, ready flags, split-K planes) comes from a
    # pool and is reused by the next call of the same shape.  Alternating two problems of one
    # shape, every result must still be its own problem's: a part of the copies that a call
    # failed to write, or a flag it failed to set, would surface as the other problem's values
    # (or as a timeout).
    M, N, K = shape
    probs = [synth.problem(M, N, K, seed=s, dist="int3") for s in (31, 32)]
    wants = [oracle.gemm(A, B, C, 1.0, -1.0, f16_inputs=True, want_mag=False)[0] for A, B, C in probs]
    for i in (0, 1, 0, 1):
        A, B, C = probs[i]
        st, got = run_cuda(phx.VARIANT_F16TC, A, B, C, 1.0, -1.0)
        assert st == phx.PHX_OK, phx.status_string(st)
        assert_bits_equal(got, wants[i], f"f16tc {shape} problem {i}")


def test_tiling_does_not_change_values():
    # Every configuration computes the same products; only how the k sums are grouped may
    # differ (one k-ordered chain per element, or, where a grid is split along K or its last
    # wave is spread over the GPU as k ranges, a few k-ordered partial sums added in k
    # order).  So on integer inputs, where every partial sum is exact, every configuration
    # gives the same bits, and on uniform inputs each stays within the bound of the oracle.
    # (The skinny configuration is tested on its own.)
    M, N, K = 2048, 2048, 1000
    Ai, Bi, Ci = synth.problem(M, N, K, seed=23, dist="int3")
    Au, Bu, Cu = synth.problem(M, N, K, seed=24, dist="uniform")
    for vname, (variant, f16) in VARIANTS.items():
        want, mag = oracle.gemm(Au, Bu, Cu, 1.0, 0.5, f16_inputs=f16)
        ref = None
        for cfg in phx.config_names(variant):
            if cfg == "SKINNY":
                continue
            phx.set_config(variant, cfg)
            got = run_cuda(variant, Ai, Bi, Ci, 1.0, 0.5)[1]
            if ref is None:
                ref = got
            else:
                assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), (vname, cfg)
            got = run_cuda(variant, Au, Bu, Cu, 1.0, 0.5)[1]
            assert_within_bound(got, want, mag, Cu, K, 1.0, 0.5, f"{vname} {cfg}")
        phx.set_config(variant, None)


# ----------------------------------------------------------------------------------------
# The tensor-core kernel's TMA epilogue (f32 C with rows 16 bytes apart): ragged M with
# whole warps of a tile past the edge, half-width tail tiles, beta = 0 and != 0, and a C
# pointer that is only 4-byte aligned (the register-path epilogue instead)
# ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(4000, 4096, 512),    # the last tile row: warps 1..3 past M
                                   (1000, 2048, 320),    # 8 x 8 pair tiles: a half-width tail round
                                   (300, 132, 100),      # N % 32 != 0 (a chunk past the edge)
                                   (2304, 2304, 1024)])  # 9 x 9 pair tiles
def test_tc_tma_epilogue(shape):
    M, N, K = shape
    _check("f16tc", M, N, K, 1.5, 0.5, "int3", seed=41)
    _check("f16tc", M, N, K, 2.0, -1.0, "uniform", seed=42)
    _check("f16tc", M, N, K, 1.0, 0.0, "int3", seed=43)


def test_tc_epilogue_unaligned_c():
    import torch
    M, N, K = 512, 256, 128
    A, B, C = synth.problem(M, N, K, seed=44, dist="int3")
    want, _ = oracle.gemm(A, B, C, 1.5, 0.5, f16_inputs=True)
    flat = torch.zeros(M * N + 1)
    flat[1:] = torch.from_numpy(C.reshape(-1))
    dC = flat.cuda()
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    st = phx.phx_gemm_f16tc_f32acc(M, N, K, 1.5, dA.data_ptr(), dB.data_ptr(), 0.5, dC.data_ptr() + 4,
                                   torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == phx.PHX_OK
    assert_bits_equal(dC.cpu().numpy()[1:].reshape(M, N), want, "C 4-byte aligned")


# ----------------------------------------------------------------------------------------
# The f32 kernel's vector edge path: M or N (or K) not a whole number of tiles, but rows 16
# bytes apart (K % 4 == N % 4 == 0, 16-byte aligned bases), so the copies stay 16 bytes wide
# and zero-fill past the edges.  Both it and the scalar edge path, which the same operands
# take when they start 4 bytes past a 16-byte boundary, against the oracle (the two kernels
# may differ in occupancy, and so in how a small grid's k sums are grouped).
# ----------------------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [(301, 260, 200), (129, 132, 20), (2000, 2048, 512), (1000, 1000, 8000),
                                   (60, 4096, 1024), (49, 4, 4), (250, 4, 1000)])
def test_sgemm_vector_edge_path(shape):
    import torch
    M, N, K = shape
    for dist, seed in (("int3", 41), ("uniform", 42)):
        A, B, C = synth.problem(M, N, K, seed=seed, dist=dist)
        want, mag = oracle.gemm(A, B, C, 1.5, -0.5, f16_inputs=False)
        out = {}
        for offset in (0, 1):
            def dev(x):
                flat = torch.zeros(x.size + 4, dtype=torch.float32)
                flat[offset:offset + x.size] = torch.from_numpy(np.ascontiguousarray(x).reshape(-1))
                return flat.cuda()
            dA, dB, dC = dev(A), dev(B), dev(C)
            st = phx.phx_sgemm(M, N, K, 1.5, dA.data_ptr() + 4 * offset, dB.data_ptr() + 4 * offset, -0.5,
                               dC.data_ptr() + 4 * offset, torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            assert st == phx.PHX_OK, phx.status_string(st)
            out[offset] = dC.cpu().numpy()[offset:offset + M * N].reshape(M, N)
        for offset, path in ((0, "vector"), (1, "scalar")):
            what = f"sgemm edges {shape} {dist} ({path})"
            if dist == "int3":
                assert_bits_equal(out[offset], want, what)
            else:
                assert_within_bound(out[offset], want, mag, C, K, 1.5, -0.5, what)


@pytest.mark.parametrize("shape,offset_a", [((1031, 1029, 4100), 0),   # N % 4 != 0: B padded
                                            ((1030, 1024, 4099), 0),   # K % 4 != 0: A and B padded
                                            ((1024, 1024, 4096), 1)])  # A not 16-byte aligned: A padded
def test_sgemm_padded_copies_of_unaligned_operands(shape, offset_a):
    # Large f32 problems whose rows of A or B do not start on 16 bytes are computed on
    # zero-padded 16-byte-aligned copies of A and/or B; C (rows unaligned too) is written in
    # place.  Bit for bit on integer inputs, within the bound on uniform ones.
    import torch
    M, N, K = shape
    for dist in ("int3", "uniform"):
        A, B, C = synth.problem(M, N, K, seed=41, dist=dist)
        want, mag = oracle.gemm(A, B, C, 1.5, -0.5)
        buf = torch.zeros(M * K + 4, device="cuda")
        dA = buf[offset_a:offset_a + M * K].view(M, K)
        dA.copy_(torch.from_numpy(A))
        dB = torch.from_numpy(B).cuda()
        dC = torch.from_numpy(C.copy()).cuda()
        st = phx.phx_sgemm(M, N, K, 1.5, dA.data_ptr(), dB.data_ptr(), -0.5, dC.data_ptr(),
                           torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert st == phx.PHX_OK
        got = dC.cpu().numpy()
        if dist == "int3":
            assert_bits_equal(got, want, f"padded {shape} {dist}")
        else:
            assert_within_bound(got, want, mag, C, K, 1.5, -0.5, f"padded {shape} {dist}")
