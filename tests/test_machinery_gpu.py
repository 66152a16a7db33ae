"""The library's machinery on a GB300: the bounded-wait timeout path, the autotuner (with
an injected failing candidate), the roof probes, and concurrent streams sharing the
workspace pool."""
import os

import numpy as np
import pytest

import oracle
from dense_gemm_04_gb300 import phx, synth
from tests.gpu_util import VARIANTS, assert_bits_equal, run_cuda

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    import torch
    s = torch.cuda.current_stream().cuda_stream
    assert phx.check_device_status() == phx.PHX_OK
    assert phx.phx_selftest_bounded_wait(1_000_000, s) == phx.PHX_OK   # 1 ms limit
    assert phx.check_device_status() == phx.PHX_ERR_TIMEOUT
    assert phx.check_device_status() == phx.PHX_OK                       # the word was cleared
    # the context is still usable
    A, B, C = synth.problem(64, 64, 64, dist="int3")
    want, _ = oracle.gemm(A, B, C, 1.0, 1.0)
    st, got = run_cuda(phx.VARIANT_SGEMM, A, B, C, 1.0, 1.0)
    assert st == phx.PHX_OK
    assert_bits_equal(got, want)


@pytest.mark.parametrize("vname", list(VARIANTS))
def test_autotune_and_injected_failure(vname, monkeypatch):
    variant, f16 = VARIANTS[vname]
    M, N, K = 768, 512, 320
    phx.set_config(variant, None)
    monkeypatch.delenv("PHX_TUNE_FAIL", raising=False)
    first = phx.autotune(variant, M, N, K, finalists=3, rounds=3, settle_ms=20)
    assert first in phx.config_names(variant)
    # the chosen configuration "fails to launch": the tuner must skip it and pick another
    monkeypatch.setenv("PHX_TUNE_FAIL", first)
    second = phx.autotune(variant, M, N, K, finalists=3, rounds=3, settle_ms=20)
    assert second != first and second in phx.config_names(variant)
    # the tuned choice is used by later calls of this shape and is correct
    assert phx.get_config(variant, M, N, K) == second
    A, B, C = synth.problem(M, N, K, dist="int3")
    want, _ = oracle.gemm(A, B, C, 1.5, 0.5, f16_inputs=f16)
    st, got = run_cuda(variant, A, B, C, 1.5, 0.5)
    assert st == phx.PHX_OK
    assert_bits_equal(got, want)


def test_probes_run():
    import torch
    s = torch.cuda.current_stream().cuda_stream
    out = torch.zeros(64 * 256, device="cuda")
    for packed in (0, 1):
        assert phx.phx_probe_ffma(packed, 64, 1000, out.data_ptr(), s) == phx.PHX_OK
        torch.cuda.synchronize()
        assert torch.isfinite(out).all() and (out > 0).all()
    # the read probe's per-block XOR folds combine to the XOR of every word of the buffer
    # (a ragged length, so the last block's slice is short)
    n = (1 << 20) + 4 * 37
    words = np.random.default_rng(3).integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
    x = torch.from_numpy(words.view(np.float32)).cuda()
    fold = torch.zeros(256, dtype=torch.int32, device="cuda")
    assert phx.phx_probe_stream_read(x.data_ptr(), n, fold.data_ptr(), 256, s) == phx.PHX_OK
    torch.cuda.synchronize()
    assert np.bitwise_xor.reduce(fold.cpu().numpy().view(np.uint32)) == np.bitwise_xor.reduce(words)
    sink_mma = torch.full((8,), 7.0, device="cuda")
    for n in (64, 128, 256):
        assert phx.phx_probe_mma_f16(8, 100, n, sink_mma.data_ptr(), s) == phx.PHX_OK
        torch.cuda.synchronize()
        assert (sink_mma == 0).all()          # zero operands give a zero accumulator
    assert phx.check_device_status() == phx.PHX_OK


def test_concurrent_streams_share_the_workspace_pool():
    import torch
    shapes = [(300, 200, 150), (257, 129, 513)]
    probs = [synth.problem(*s, seed=i, dist="int3") for i, s in enumerate(shapes)]
    wants = [oracle.gemm(A, B, C, 1.0, 1.0, f16_inputs=True)[0] for A, B, C in probs]
    streams = [torch.cuda.Stream() for _ in shapes]
    dev = [[torch.from_numpy(x).cuda() for x in p] for p in probs]
    torch.cuda.synchronize()
    outs = [[] for _ in shapes]
    for rep in range(8):
        for i, ((M, N, K), (dA, dB, dC), st) in enumerate(zip(shapes, dev, streams)):
            with torch.cuda.stream(st):
                c = dC.clone()
                assert phx.phx_gemm_f16tc_f32acc(M, N, K, 1.0, dA.data_ptr(), dB.data_ptr(), 1.0,
                                                 c.data_ptr(), st.cuda_stream) == phx.PHX_OK
                outs[i].append(c)
    torch.cuda.synchronize()
    for i in range(len(shapes)):
        for c in outs[i]:
            assert_bits_equal(c.cpu().numpy(), wants[i])


@pytest.mark.gpu
def test_last_config_reports_what_ran():
    import torch
    from dense_gemm_04_gb300 import phx
    A = torch.rand(512, 512, device="cuda")
    C = torch.zeros(512, 512, device="cuda")
    for variant, fn in ((phx.VARIANT_SGEMM, phx.sgemm), (phx.VARIANT_F16TC, phx.gemm_f16tc_f32acc)):
        phx.set_config(variant, None)
        fn(A, A, C)
        assert phx.last_config(variant) == phx.get_config(variant, 512, 512, 512)
        fn(A[:8].contiguous(), A, C[:8].contiguous())   # few rows: the skinny kernel
        assert phx.last_config(variant) == "SKINNY"
