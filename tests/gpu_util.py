"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on seeded inputs
and compare with the oracle."""
import numpy as np

from dense_gemm_04_gb300 import phx

VARIANTS = {"sgemm": (phx.VARIANT_SGEMM, False), "f16tc": (phx.VARIANT_F16TC, True)}


def bound(mag, C, K, alpha, beta):
    """Per-element bound 8 * sqrt(K) * 2^-24 * (|alpha| * sum_k |a||b| + |beta| * |C|): the
    tolerance stated for both precisions (f16 x f16 products are exact in f32, so the
    tensor-core path rounds only in its f32 sums, like the f32 path)."""
    return 8.0 * np.sqrt(max(K, 1)) * 2.0 ** -24 * (abs(alpha) * mag + abs(beta) * np.abs(C.astype(np.float64)))


def run_cuda(variant, A, B, C, alpha, beta, stream=None):
    """C-ABI call on device copies of the numpy inputs; returns (status, result as numpy)."""
    import torch
    M, K = A.shape
    N = B.shape[1]
    dA = torch.from_numpy(np.ascontiguousarray(A)).cuda()
    dB = torch.from_numpy(np.ascontiguousarray(B)).cuda()
    dC = torch.from_numpy(np.ascontiguousarray(C)).cuda()
    fn = phx.phx_sgemm if variant == phx.VARIANT_SGEMM else phx.phx_gemm_f16tc_f32acc
    h = torch.cuda.current_stream().cuda_stream if stream is None else stream
    st = fn(M, N, K, alpha, dA.data_ptr(), dB.data_ptr(), beta, dC.data_ptr(), h)
    torch.cuda.synchronize()
    return st, dC.cpu().numpy()


def assert_within_bound(got, want, mag, C, K, alpha, beta, what=""):
    tol = bound(mag, C, K, alpha, beta)
    err = np.abs(got.astype(np.float64) - want.astype(np.float64))
    bad = ~(err <= tol)  # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = [(tuple(int(v) for v in i), float(got[tuple(i)]), float(want[tuple(i)]), float(tol[tuple(i)]))
                  for i in idx]
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside the bound, e.g. {detail}")


def assert_bits_equal(got, want, what=""):
    g = got.view(np.uint32)
    w = want.view(np.uint32)
    # +0 and -0 both mean zero (the sign of a zero sum depends on the summation order)
    same = (g == w) | ((got == 0) & (want == 0))
    if not same.all():
        idx = np.argwhere(~same)[:5]
        detail = [(tuple(int(v) for v in i), float(got[tuple(i)]), float(want[tuple(i)])) for i in idx]
        raise AssertionError(f"{what}: {int((~same).sum())} elements differ, e.g. {detail}")
