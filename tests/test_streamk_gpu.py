"""Stream-K schedules of the f32 GEMM on a GB300, through phx_sgemm, against the oracle.

A grid whose last wave would leave SMs idle -- or a grid of less than one wave -- spreads the
k tiles of that wave's tiles evenly over stream-K blocks; each such tile is then the sum, in
k order, of a few partial tiles ("gemm, f32", sections "One output tile per CTA" and
"Tuning": the same products, only split along k).  With the 128 x 128 tile (two CTAs per
SM, 304 slots on 152 SMs) the shapes below give: tails of 20, 38 and 176 tiles after whole
waves, aligned and masked; and whole grids of 4, 16, 64 (masked) and 128 tiles spread over
8 to 304 blocks.  Integer inputs must match the oracle bit for bit (every partial sum is
exact), uniform ones within 8 * sqrt(K) * 2^-24 * (|alpha| sum|a||b| + |beta||C|).
"""
import numpy as np
import pytest

import oracle
from dense_gemm_04_gb300 import phx, synth
from tests.gpu_util import assert_bits_equal, assert_within_bound, run_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _status():
    phx.set_config(phx.VARIANT_SGEMM, None)
    yield
    phx.set_config(phx.VARIANT_SGEMM, None)
    assert phx.check_device_status() == phx.PHX_OK


def _check(M, N, K, alpha, beta, dist, seed):
    A, B, C = synth.problem(M, N, K, seed=seed, dist=dist)
    want, mag = oracle.gemm(A, B, C, alpha, beta, f16_inputs=False)
    st, got = run_cuda(phx.VARIANT_SGEMM, A, B, C, alpha, beta)
    assert st == phx.PHX_OK, phx.status_string(st)
    what = f"stream-K sgemm {(M, N, K)} {dist} [{phx.last_config(phx.VARIANT_SGEMM)}]"
    if dist == "int3":
        assert_bits_equal(got, want, what)
    else:
        assert_within_bound(got, want, mag, C, K, alpha, beta, what)
    return got


@pytest.mark.parametrize("shape", [(2304, 2304, 2048), (2300, 2310, 2000), (4096, 4352, 512),
                                   (256, 256, 256), (512, 512, 512), (1000, 1000, 8000), (16384, 128, 4096)])
def test_streamk_parity(shape):
    M, N, K = shape
    _check(M, N, K, 1.5, 0.5, "int3", seed=31)
    _check(M, N, K, 2.0, -1.0, "uniform", seed=32)


def test_streamk_one_cta_per_sm_config():
    # a tile of 128 x 256 (one CTA per SM): 162 tiles on 152 slots, a tail of 10
    phx.set_config(phx.VARIANT_SGEMM, "TILE_M=128 TILE_N=256 TILE_K=16 STAGES=4 FMA2=1")
    _check(2304, 2304, 2048, 1.0, 0.0, "int3", seed=33)
    _check(2304, 2304, 2048, 1.0, 0.5, "uniform", seed=34)


def test_streamk_special_values_and_determinism():
    M, N, K = 2304, 2304, 2048
    A, B, C = synth.problem(M, N, K, seed=35, dist="uniform")
    # beta == 0 with NaN in C: C is not read, in the whole-tile part and in the tail
    st, got = run_cuda(phx.VARIANT_SGEMM, A, B, np.full_like(C, np.nan), 1.0, 0.0)
    assert st == phx.PHX_OK and np.isfinite(got).all()
    # the same call twice: the same bits (the split of the tail depends on the shape only)
    _, r1 = run_cuda(phx.VARIANT_SGEMM, A, B, C, 1.0, 0.5)
    _, r2 = run_cuda(phx.VARIANT_SGEMM, A, B, C, 1.0, 0.5)
    assert_bits_equal(r1, r2, "two runs")


def test_profile_counts_the_kernels_of_each_schedule():
    # on 152 SMs with the 128 x 128 tile: whole waves plus a tail spread as stream-K blocks
    # launch three kernels (stream-K blocks, fix-up, whole tiles); one wave of tiles, one; a
    # grid split along K, two (the slices and their reduction); a grid spread whole as
    # stream-K blocks, two (the blocks and the fix-up)
    import torch
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the schedules below are those of a 152-SM GPU")
    for shape, kernels in (((2304, 2304, 2048), 3), ((2048, 2048, 256), 1), ((1024, 1024, 1024), 2),
                           ((128, 128, 16384), 2)):
        M, N, K = shape
        A, B, C = synth.problem(M, N, K, seed=36, dist="int3")
        phx.profile_start()
        st, got = run_cuda(phx.VARIANT_SGEMM, A, B, C, 1.0, 0.5)
        prof = phx.profile_stop()
        assert st == phx.PHX_OK
        assert prof["sgemm"][0] == kernels, (shape, prof["sgemm"])
        want, _ = oracle.gemm(A, B, C, 1.0, 0.5, f16_inputs=False)
        assert_bits_equal(got, want, f"{shape}")
