"""The allocation-free variant of the f16 tensor-core GEMM, through the C ABI.

phx_gemm_f16tc_f32acc_noalloc exists for callers that cannot allocate device memory while
they run (a latency-critical loop that must not wait on an allocator, or a plug-in whose
host application owns the device-memory budget).  It keeps its scratch, the f16 copies of A
and B, in the library's 64 MiB static device array instead of a pooled workspace.  It must
give the results of phx_gemm_f16tc_f32acc, call after call, although every call reuses the
same array; and it must refuse problems whose scratch would not fit.

This file is collected after every other test file, so a run that stops at the first failure
has already run the rest.  It passes alone in a fresh process (its first call does the
per-device set-up) and after the other tests.
"""
import numpy as np
import pytest

import oracle
from dense_gemm_04_gb300 import phx, synth
from tests.gpu_util import assert_within_bound

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


def test_noalloc_matches_the_pooled_entry_point_call_after_call():
    phx.set_config(phx.VARIANT_F16TC, None)
    problems = [
        (1000, 900, 700, 1.5, 0.5, 11),      # ragged in every dimension
        (2048, 1536, 2048, 1.0, 0.5, 12),    # a larger problem reusing the same scratch
        (1000, 900, 700, 1.5, 0.5, 13),      # back to the first shape: stale scratch is harmless
        (8, 4096, 4096, 1.0, 0.5, 14),       # few rows of A: the skinny kernel, K split in a cluster
        (2, 128, 65536, 1.0, 0.5, 15),       # ... and in planes of partial sums in the scratch
    ]
    for M, N, K, alpha, beta, seed in problems:
        A, B, C = synth.problem(M, N, K, seed=seed)
        st_ref, want = _call(phx.phx_gemm_f16tc_f32acc, A, B, C, alpha, beta)
        st, got = _call(phx.phx_gemm_f16tc_f32acc_noalloc, A, B, C, alpha, beta)
        assert st_ref == phx.PHX_OK and st == phx.PHX_OK, (phx.status_string(st_ref), phx.status_string(st))
        _, mag = oracle.gemm(A, B, C, alpha, beta, f16_inputs=True)
        assert_within_bound(got, want, mag, C, K, alpha, beta, f"noalloc {(M, N, K)}")
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
