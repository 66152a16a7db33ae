"""The allocation-free variant of the f16 tensor-core GEMM, through the C ABI.

phx_gemm_f16tc_f32acc_noalloc exists for callers that cannot allocate device memory while
they run (a latency-critical loop that must not wait on an allocator, or a plug-in whose
host application owns the device-memory budget).  It keeps its scratch, the f16 copies of A
and B and any split-K planes, in the library's 64 MiB static device array instead of a pooled
workspace.  Its results must match the oracle (within the bound, and bit for bit on
integer-valued inputs) and equal those of phx_gemm_f16tc_f32acc bit for bit, call after
call, although every call reuses the same array; it must refuse problems whose scratch would
not fit; and a bounded wait that gives up inside it must be reported by
phx_check_device_status.

This file is collected after every other test file, so a run that stops at the first failure
has already run the rest.  It passes alone in a fresh process (its first call does the
per-device set-up) and after the other tests.
"""
import numpy as np
import pytest

import oracle
from dense_gemm_04_gb300 import phx, synth
from tests.gpu_util import assert_bits_equal, assert_within_bound

pytestmark = pytest.mark.gpu


def _call(fn, A, B, C, alpha, beta):
    import torch
    M, K = A.shape
    N = B.shape[1]
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C.copy()).cuda()
    st = fn(M, N, K, alpha, dA.data_ptr(), dB.data_ptr(), beta, dC.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return st, dC.cpu().numpy()


PROBLEMS = [
    (1000, 900, 700, 1.5, 0.5, 11),      # ragged in every dimension
    (2048, 1536, 2048, 1.0, 0.5, 12),    # a larger problem reusing the same scratch
    (1000, 900, 700, 1.5, 0.5, 13),      # back to the first shape: stale scratch is harmless
    (512, 512, 8192, 2.0, -1.0, 16),     # a grid too small for the GPU: split-K planes in the array
    (8, 4096, 4096, 1.0, 0.5, 14),       # few rows of A: the skinny kernel, K split in a cluster
    (2, 128, 65536, 1.0, 0.5, 15),       # ... and in planes of partial sums in the scratch
    (8, 8192, 4096, 1.0, 0.5, 17),       # skinny: more than 64 MiB of f16 copies, which it never makes
    (16384, 128, 1024, 1.0, 0.5, 18),    # few columns: A rounded inside the GEMM, only B's copy in the array
    (64, 4096, 4096, 1.0, 0.5, 19),      # few rows: B rounded inside the GEMM, A's copy and K-split planes
    (2085, 96, 4100, 2.0, -1.0, 20),     # fewer row tiles than SMs: A rounded inside, B's copy and K-split planes
    (4096, 3, 4096, 1.0, 0.5, 21),       # few columns: the skinny kernel on the transposed product
]


@pytest.mark.parametrize("dist", ["uniform", "int3"])
def test_noalloc_matches_the_oracle_call_after_call(dist):
    phx.set_config(phx.VARIANT_F16TC, None)
    assert phx.check_device_status() == phx.PHX_OK
    for M, N, K, alpha, beta, seed in PROBLEMS:
        A, B, C = synth.problem(M, N, K, seed=seed, dist=dist)
        want, mag = oracle.gemm(A, B, C, alpha, beta, f16_inputs=True)
        # two calls in a row on the same inputs: the second one finds the first one's scratch
        for rep in range(2):
            st, got = _call(phx.phx_gemm_f16tc_f32acc_noalloc, A, B, C, alpha, beta)
            assert st == phx.PHX_OK, phx.status_string(st)
            what = f"noalloc {(M, N, K)} {dist} call {rep}"
            if dist == "int3":
                assert_bits_equal(got, want, what)      # every partial sum is an exact integer
            else:
                assert_within_bound(got, want, mag, C, K, alpha, beta, what)
        # the pooled entry point runs the same schedule: the same bits
        st_ref, pooled = _call(phx.phx_gemm_f16tc_f32acc, A, B, C, alpha, beta)
        assert st_ref == phx.PHX_OK
        assert_bits_equal(got, pooled, f"noalloc vs pooled {(M, N, K)} {dist}")
    assert phx.check_device_status() == phx.PHX_OK


def test_noalloc_refuses_problems_beyond_its_scratch():
    import torch
    # (4096 + 4097) rows of 4096 halves need more than 64 MiB of scratch
    M, N, K = 4096, 4097, 4096
    assert phx.f16tc_workspace_bytes(M, N, K) > 64 << 20
    assert phx.f16tc_workspace_bytes(4096, 4096, 4096) <= 64 << 20
    A = torch.zeros((M, K), device="cuda")
    B = torch.zeros((K, N), device="cuda")
    C = torch.full((M, N), 3.0, device="cuda")
    st = phx.phx_gemm_f16tc_f32acc_noalloc(M, N, K, 1.0, A.data_ptr(), B.data_ptr(), 0.0,
                                           C.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == phx.PHX_ERR_NOMEM
    assert bool((C == 3.0).all())


def test_noalloc_timeout_is_reported_and_cleared():
    import torch
    s = torch.cuda.current_stream().cuda_stream
    assert phx.check_device_status() == phx.PHX_OK
    # a wait on a barrier nothing arrives at, 1 ms limit, recorded in the static array's word
    assert phx.phx_selftest_bounded_wait_noalloc(1_000_000, s) == phx.PHX_OK
    assert phx.check_device_status() == phx.PHX_ERR_TIMEOUT
    assert phx.check_device_status() == phx.PHX_OK          # the word was cleared
    # the context still works: a GEMM through the same array afterwards
    A, B, C = synth.problem(300, 200, 150, seed=5, dist="int3")
    want, _ = oracle.gemm(A, B, C, 1.0, 1.0, f16_inputs=True)
    st, got = _call(phx.phx_gemm_f16tc_f32acc_noalloc, A, B, C, 1.0, 1.0)
    assert st == phx.PHX_OK
    assert_bits_equal(got, want, "noalloc after a timeout")
    assert phx.check_device_status() == phx.PHX_OK
