"""Runs shapes that exercise every schedule of libphx through its bounds-checked build (the
library PHX_LIBRARY names, built with PHX_DEBUG=1) and checks each result against the oracle,
then prints the number of failed index checks.  Started by tests/test_debug_build_gpu.py in
a process of its own, so that the binding loads that library.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from dense_gemm_04_gb300 import phx, synth  # noqa: E402

EDGE_DIMS = [1, 2, 3, 15, 16, 17, 63, 64, 65, 127, 128, 129]


def run(variant, f16, M, N, K, alpha, beta, seed):
    import torch
    A, B, C = synth.problem(M, N, K, seed=seed, dist="int3")
    want, _ = oracle.gemm(A, B, C, alpha, beta, f16_inputs=f16, want_mag=False)
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C.copy()))
    fn = phx.phx_sgemm if variant == phx.VARIANT_SGEMM else phx.phx_gemm_f16tc_f32acc
    st = fn(M, N, K, alpha, dA.data_ptr(), dB.data_ptr(), beta, dC.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    got = dC.cpu().numpy()
    same = (got.view(np.uint32) == want.view(np.uint32)) | ((got == 0) & (want == 0))
    return st == phx.PHX_OK and bool(same.all())


def main():
    assert phx.phx_debug_build() == 1, "PHX_LIBRARY must name the bounds-checked build"
    rng = np.random.default_rng(5)
    shapes = {(d, d, d) for d in EDGE_DIMS}
    for _ in range(40):
        shapes.add(tuple(int(x) for x in rng.choice(EDGE_DIMS, 3)))
    # the schedules: stream-K tail and whole-grid stream-K, split-K, the TMA epilogue, half-width
    # tail items, the skinny kernels (few rows), ragged and padded edges
    shapes |= {(256, 256, 256), (1024, 1024, 4096), (300, 500, 3000), (2048, 2048, 256), (3000, 2000, 700),
               (8, 4096, 4096), (2, 128, 65536), (40, 1000, 3000), (1031, 1029, 4100), (1030, 1024, 4099),
               (10000, 100, 300), (64, 3000, 2000)}  # few columns / few rows (the kernel that rounds A / B)
    # few columns against many rows: the skinny kernel on the transposed product (default routes)
    narrow = [(2085, 7, 2050), (1024, 3, 65536)]
    failures = []
    runs = 0
    for variant, f16 in ((phx.VARIANT_SGEMM, False), (phx.VARIANT_F16TC, True)):
        for i, (M, N, K) in enumerate(sorted(shapes) + narrow):
            runs += 1
            if not run(variant, f16, M, N, K, 1.5, 0.5, i):
                failures.append((variant, M, N, K))
    # the kernel that rounds A or B, pinned, on the edge shapes
    for cfg in [n for n in phx.config_names(phx.VARIANT_F16TC) if "CONVERT" in n]:
        phx.set_config(phx.VARIANT_F16TC, cfg)
        for i, (M, N, K) in enumerate(sorted(shapes)):
            if M * N * K > 2 ** 31:
                continue
            runs += 1
            if not run(phx.VARIANT_F16TC, True, M, N, K, 1.5, 0.5, 100 + i):
                failures.append((cfg, M, N, K))
        phx.set_config(phx.VARIANT_F16TC, None)
    count = phx.debug_violations()
    print(f"shapes {runs} failures {len(failures)} violations {count}")
    if failures:
        print("failed:", failures[:10])
    return 0 if not failures and count == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
