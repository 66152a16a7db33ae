"""Shape and arithmetic-intensity sweep of both GEMM precisions, placed on the roofline.

    python -m dense_gemm_04_gb300.sweep [--out results.json] [--quick] [--layouts] [--skinny] [--narrow]
        [--f16in]
    python -m dense_gemm_04_gb300.sweep --one M,N,K [--variant sgemm|f16tc|f16in|f16out] [--calls 5]
        [--alpha 1] [--beta 0] [--b-transposed]

For every shape of the workload sweep ((8192, 8192, 1024), (1024, 1024, 16384),
(16384, 128, 4096), (4095, 4097, 4093) with alpha = 2, beta = -1; squares 512 .. 16384 with
alpha = 1, beta = 0; and 4096^3 with alpha = 1, beta = 0.5) and both precisions, this measures
the GEMM the way the matrix-multiplication lab's stopwatches do: settle the clock with synced
calls, then take the median of CUDA-event timings ("steady"), with the shapes visited in a
freshly shuffled order every round ("sweep").  Beside each steady time it reports the host
microseconds spent inside one call and the GPU time per call with 50 calls queued back to
back (no host gaps).  Each result is placed on its roofline,
min(peak, bandwidth x intensity), with intensity = 2MNK / minimum bytes (each f32 input
read once, C written once and read when beta != 0), following the lab's minimum-traffic
intensity (Part 5, the skinny-matrix sweep).

The roofs are measured here as well: the FP32 multiply-add probe and the tensor-core probe
run back to back for two seconds each while nvidia-smi samples the clocks (the lab's
"sustained"), next to a streaming-read probe.  Inputs are synthetic uniform [-1, 1) matrices.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

from . import phx

SHAPES = [
    ("4096^3", 4096, 4096, 4096, 1.0, 0.5),
    ("8192x8192x1024", 8192, 8192, 1024, 2.0, -1.0),
    ("1024x1024x16384", 1024, 1024, 16384, 2.0, -1.0),
    ("16384x128x4096", 16384, 128, 4096, 2.0, -1.0),
    ("4095x4097x4093", 4095, 4097, 4093, 2.0, -1.0),
] + [(f"{n}^3", n, n, n, 1.0, 0.0) for n in (512, 1024, 2048, 4096, 8192, 16384)]


class Clocks:
    """nvidia-smi SM clock and power samples every 200 ms while active."""

    def __init__(self, gpu: int = 0):
        self.gpu, self.samples, self._stop = gpu, [], threading.Event()

    def _loop(self):
        while not self._stop.is_set():
            try:
                out = subprocess.run(["nvidia-smi", "-i", str(self.gpu),
                                      "--query-gpu=clocks.sm,power.draw,clocks_event_reasons.active",
                                      "--format=csv,noheader,nounits"],
                                     capture_output=True, text=True, timeout=5).stdout.strip()
                p = [x.strip() for x in out.split(",")]
                self.samples.append((float(p[0]), float(p[1]), p[2]))
            except (OSError, ValueError, IndexError, subprocess.TimeoutExpired):
                pass
            self._stop.wait(0.2)

    def __enter__(self):
        self._t = threading.Thread(target=self._loop, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        self._t.join()

    def summary(self):
        if not self.samples:
            return {}
        sm = sorted(s[0] for s in self.samples)
        return {"sm_mhz_median": sm[len(sm) // 2], "power_w_max": max(s[1] for s in self.samples),
                "samples": len(sm), "reasons": sorted({s[2] for s in self.samples})}


def _sync():
    import torch
    torch.cuda.synchronize()


def steady(fn, seconds=0.5, min_calls=3):
    """Median seconds per call after settling for seconds/2 with one synced call at a time."""
    import torch
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds / 2:
        fn()
        _sync()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ts, t0 = [], time.perf_counter()
    while time.perf_counter() - t0 < seconds or len(ts) < min_calls:
        s.record()
        fn()
        e.record()
        e.synchronize()
        ts.append(s.elapsed_time(e) / 1e3)
    return float(np.median(ts))


def host_and_queued(fn, queue=50):
    """(median host seconds spent inside one call, GPU seconds per call with `queue` calls
    queued back to back between two events).  The first is the library's own cost on the
    host: argument checks, the configuration lookup and the launches, without waiting for
    the GPU.  The second is the device time per call without the host's gaps between calls."""
    import torch
    fn()
    _sync()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    host = []
    ev0.record()
    for _ in range(queue):
        t0 = time.perf_counter()
        fn()
        host.append(time.perf_counter() - t0)
    ev1.record()
    ev1.synchronize()
    return float(np.median(host)), ev0.elapsed_time(ev1) / 1e3 / queue


def sustained(fn, seconds=2.0):
    """Seconds per call under continuous load, with the clocks it ran at."""
    import torch
    fn()
    _sync()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks() as clk:
        s.record()
        n, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            fn()
            n += 1
            if n % 4 == 0:
                _sync()
        e.record()
        e.synchronize()
    return s.elapsed_time(e) / 1e3 / n, clk.summary()


def measure_roofs(seconds=2.0):
    import torch
    dev = torch.cuda.current_device()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    st = torch.cuda.current_stream().cuda_stream
    roofs = {"sms": sms}
    blocks, iters = sms * 8 * 8, 20000
    out = torch.empty(blocks * 256, device="cuda")
    for packed in (0, 1):
        t, clk = sustained(lambda: phx.check(phx.phx_probe_ffma(packed, blocks, iters, out.data_ptr(), st)), seconds)
        roofs["fp32_ffma2" if packed else "fp32_ffma"] = {
            "tflops": blocks * 256 * iters * 24 / t / 1e12, "clocks": clk}
    sink = torch.empty(sms, device="cuda")
    t, clk = sustained(lambda: phx.check(phx.phx_probe_mma_f16(sms, 4000, 256, sink.data_ptr(), st)), seconds)
    roofs["f16_tensor"] = {"tflops": sms * 4000 * 4 * 2 * 128 * 256 * 16 / t / 1e12, "clocks": clk}
    x = torch.ones(1 << 28, device="cuda")
    fold = torch.empty(sms * 8, dtype=torch.int32, device="cuda")
    t = steady(lambda: phx.check(phx.phx_probe_stream_read(x.data_ptr(), x.numel(), fold.data_ptr(), sms * 8, st)))
    roofs["hbm_read_gbs"] = x.numel() * 4 / t / 1e9
    del x
    return roofs


def run(quick=False, rounds=3, seed=0):
    import torch
    st = torch.cuda.current_stream().cuda_stream
    roofs = measure_roofs(1.0 if quick else 2.0)
    fp32 = max(roofs["fp32_ffma"]["tflops"], roofs["fp32_ffma2"]["tflops"])
    tc = roofs["f16_tensor"]["tflops"]
    bw = roofs["hbm_read_gbs"]
    shapes = [s for s in SHAPES if not (quick and s[1] * s[2] * s[3] > 2 ** 40)]
    cases = [(s, v) for s in shapes for v in ("sgemm", "f16tc")]
    times = {c: [] for c in range(len(cases))}
    host = {c: [] for c in range(len(cases))}
    queued = {c: [] for c in range(len(cases))}
    rng = np.random.default_rng(seed)
    for _ in range(rounds):
        for ci in rng.permutation(len(cases)):
            (name, M, N, K, alpha, beta), v = cases[ci]
            A = torch.rand(M, K, device="cuda") * 2 - 1
            B = torch.rand(K, N, device="cuda") * 2 - 1
            C = torch.rand(M, N, device="cuda") * 2 - 1
            fn = phx.phx_sgemm if v == "sgemm" else phx.phx_gemm_f16tc_f32acc
            call = lambda: phx.check(fn(M, N, K, alpha, A.data_ptr(), B.data_ptr(), beta, C.data_ptr(), st))
            times[ci].append(steady(call, seconds=0.3 if quick else 0.5))
            h, q = host_and_queued(call)
            host[ci].append(h)
            queued[ci].append(q)
            del A, B, C
            torch.cuda.empty_cache()
    rows = []
    for ci, ((name, M, N, K, alpha, beta), v) in enumerate(cases):
        t = float(np.median(times[ci]))
        flops = 2.0 * M * N * K
        nbytes = 4.0 * (M * K + K * N + M * N * (2 if beta != 0 else 1))
        ai = flops / nbytes
        peak = fp32 if v == "sgemm" else tc
        roof = min(peak * 1e12, bw * 1e9 * ai)
        rows.append({"shape": name, "M": M, "N": N, "K": K, "alpha": alpha, "beta": beta, "variant": v,
                     "config": phx.get_config(0 if v == "sgemm" else 1, M, N, K),
                     "seconds": t, "tflops": flops / t / 1e12, "intensity": ai,
                     "host_us_per_call": 1e6 * float(np.median(host[ci])),
                     "queued_seconds": float(np.median(queued[ci])),
                     "queued_tflops": flops / float(np.median(queued[ci])) / 1e12,
                     "roof_tflops": roof / 1e12, "pct_of_roof": 100 * flops / t / roof,
                     "bound": "compute" if roof >= peak * 1e12 else "hbm",
                     "seconds_all": times[ci]})
    return {"roofs": roofs, "rows": rows}


def run_layouts(n=4096, rounds=3, seed=0, seconds=0.5):
    """The lab's layout sweep (Part 5): A @ B with A, B or both stored transposed, n^3,
    alpha = 1, beta = 0, both precisions; median seconds over shuffled rounds."""
    import torch
    st = torch.cuda.current_stream().cuda_stream
    A = torch.rand(n, n, device="cuda") * 2 - 1
    B = torch.rand(n, n, device="cuda") * 2 - 1
    C = torch.zeros(n, n, device="cuda")
    At, Bt = A.t().contiguous(), B.t().contiguous()
    cases = [(v, oa, ob) for v in ("sgemm", "f16tc") for oa in (phx.OP_N, phx.OP_T) for ob in (phx.OP_N, phx.OP_T)]
    times = {c: [] for c in cases}
    rng = np.random.default_rng(seed)
    for _ in range(rounds):
        for ci in rng.permutation(len(cases)):
            v, oa, ob = cases[ci]
            fn = phx.phx_sgemm_ex if v == "sgemm" else phx.phx_gemm_f16tc_f32acc_ex
            a = (At if oa == phx.OP_T else A).data_ptr()
            b = (Bt if ob == phx.OP_T else B).data_ptr()
            times[cases[ci]].append(steady(lambda: phx.check(fn(oa, ob, n, n, n, 1.0, a, b, 0.0, C.data_ptr(), st)),
                                           seconds=seconds))
    rows = []
    for v, oa, ob in cases:
        t = float(np.median(times[(v, oa, ob)]))
        plain = float(np.median(times[(v, phx.OP_N, phx.OP_N)]))
        name = ("A.T" if oa == phx.OP_T else "A") + " @ " + ("B.T" if ob == phx.OP_T else "B")
        rows.append({"variant": v, "layout": name, "seconds": t, "tflops": 2.0 * n ** 3 / t / 1e12,
                     "vs_plain": plain / t})
    return rows


def run_skinny(rounds=3, seed=0, seconds=0.3, queue=50, b_transposed=False):
    """The lab's skinny-matrix sweep (Part 5): (M x 4096) @ (4096 x 4096) for M = 1 .. 2048,
    both precisions, alpha = 1, beta = 0, with the default configuration (the skinny kernel
    for small M).  Times are the median over shuffled rounds of `queue` back-to-back calls
    between two events (the GPU time per call, without the host's launch gaps), and the
    least traffic 4 (MK + KN + MN) bytes gives the bandwidth each call reached."""
    import torch
    st = torch.cuda.current_stream().cuda_stream
    K = N = 4096
    Ms = [1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048]
    B = torch.rand(K, N, device="cuda") * 2 - 1
    if b_transposed:   # B stored N x K, the layout of a weight matrix in x @ W^T
        B = B.t().contiguous()
    op_b = phx.OP_T if b_transposed else phx.OP_N
    X = {M: (torch.rand(M, K, device="cuda") * 2 - 1, torch.zeros(M, N, device="cuda")) for M in Ms}
    cases = [(v, M) for v in ("sgemm", "f16tc") for M in Ms]
    times = {c: [] for c in cases}
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    rng = np.random.default_rng(seed)
    for _ in range(rounds):
        for ci in rng.permutation(len(cases)):
            v, M = cases[ci]
            A, C = X[M]
            fn = phx.phx_sgemm_ex if v == "sgemm" else phx.phx_gemm_f16tc_f32acc_ex
            call = lambda: phx.check(fn(phx.OP_N, op_b, M, N, K, 1.0, A.data_ptr(), B.data_ptr(), 0.0, C.data_ptr(), st))
            t0 = time.perf_counter()
            while time.perf_counter() - t0 < seconds / 2:
                call()
                _sync()
            ev0.record()
            for _ in range(queue):
                call()
            ev1.record()
            ev1.synchronize()
            times[cases[ci]].append(ev0.elapsed_time(ev1) / 1e3 / queue)
    rows = []
    for v, M in cases:
        t = float(np.median(times[(v, M)]))
        nbytes = 4.0 * (M * K + K * N + M * N)
        rows.append({"variant": v, "M": M, "seconds": t, "tflops": 2.0 * M * N * K / t / 1e12,
                     "gbs": nbytes / t / 1e9, "intensity": 2.0 * M * N * K / nbytes,
                     "config": phx.get_config(0 if v == "sgemm" else 1, M, N, K)})
    return rows


def run_narrow(rounds=3, seed=0, seconds=0.3, queue=50):
    """The skinny sweep turned on its side: few columns of B and C.  (M x 4096) @ (4096 x N)
    for N = 1 .. 2048 at M = 4096, and N = 128 at M = 1024 .. 16384, both precisions,
    alpha = 1, beta = 0, with the default configuration (for the f16 variant, the kernel that
    rounds A inside the GEMM where A is most of the bytes).  Timed as run_skinny times: the
    median over shuffled rounds of `queue` back-to-back calls between two events; the least
    traffic 4 (MK + KN + MN) bytes gives the bandwidth each call reached."""
    import torch
    st = torch.cuda.current_stream().cuda_stream
    K = 4096
    shapes = [(4096, n) for n in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048)]
    shapes += [(m, 128) for m in (1024, 2048, 8192, 16384)]
    A = {m: torch.rand(m, K, device="cuda") * 2 - 1 for m in sorted({m for m, _ in shapes})}
    B = {n: torch.rand(K, n, device="cuda") * 2 - 1 for n in sorted({n for _, n in shapes})}
    Cs = {sh: torch.zeros(*sh, device="cuda") for sh in shapes}
    cases = [(v, sh) for v in ("sgemm", "f16tc") for sh in shapes]
    times = {c: [] for c in cases}
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    rng = np.random.default_rng(seed)
    for _ in range(rounds):
        for ci in rng.permutation(len(cases)):
            v, (M, N) = cases[ci]
            a, b, c = A[M], B[N], Cs[(M, N)]
            fn = phx.phx_sgemm if v == "sgemm" else phx.phx_gemm_f16tc_f32acc
            call = lambda: phx.check(fn(M, N, K, 1.0, a.data_ptr(), b.data_ptr(), 0.0, c.data_ptr(), st))
            t0 = time.perf_counter()
            while time.perf_counter() - t0 < seconds / 2:
                call()
                _sync()
            ev0.record()
            for _ in range(queue):
                call()
            ev1.record()
            ev1.synchronize()
            times[cases[ci]].append(ev0.elapsed_time(ev1) / 1e3 / queue)
    rows = []
    for v, (M, N) in cases:
        t = float(np.median(times[(v, (M, N))]))
        nbytes = 4.0 * (M * K + K * N + M * N)
        rows.append({"variant": v, "M": M, "N": N, "K": K, "seconds": t, "tflops": 2.0 * M * N * K / t / 1e12,
                     "gbs": nbytes / t / 1e9, "intensity": 2.0 * M * N * K / nbytes,
                     "config": phx.get_config(0 if v == "sgemm" else 1, M, N, K)})
    return rows


def run_f16in(rounds=3, seed=0, seconds=0.5):
    """Half-precision operands against the f32-operand tensor-core path (the lab's Part 4
    precision study: cuBLAS f16 GEMM), squares 2048 .. 8192 with alpha = 1, beta = 0.5:
    phx_gemm_f16tc_f32acc (f32 in, rounded in the op), phx_gemm_f16in_f32acc (f16 in, f32
    out) and phx_gemm_f16in_f16out (f16 in and out).  Median seconds of steady timing over
    shuffled rounds."""
    import torch
    st = torch.cuda.current_stream().cuda_stream
    sizes = (2048, 4096, 8192)
    kinds = ("f32in_f32out", "f16in_f32out", "f16in_f16out")
    cases = [(n, k) for n in sizes for k in kinds]
    times = {c: [] for c in cases}
    rng = np.random.default_rng(seed)
    for _ in range(rounds):
        for ci in rng.permutation(len(cases)):
            n, kind = cases[ci]
            A = torch.rand(n, n, device="cuda") * 2 - 1
            B = torch.rand(n, n, device="cuda") * 2 - 1
            C = torch.rand(n, n, device="cuda") * 2 - 1
            if kind == "f32in_f32out":
                call = lambda: phx.check(phx.phx_gemm_f16tc_f32acc(n, n, n, 1.0, A.data_ptr(), B.data_ptr(), 0.5,
                                                                   C.data_ptr(), st))
            else:
                A, B = A.half(), B.half()
                if kind == "f16in_f16out":
                    C = C.half()
                fn = phx.phx_gemm_f16in_f32acc if kind == "f16in_f32out" else phx.phx_gemm_f16in_f16out
                call = lambda: phx.check(fn(0, 0, n, n, n, 1.0, A.data_ptr(), B.data_ptr(), 0.5, C.data_ptr(), st))
            times[cases[ci]].append(steady(call, seconds=seconds))
            del A, B, C
            torch.cuda.empty_cache()
    return [{"n": n, "kind": kind, "seconds": float(np.median(times[(n, kind)])),
             "tflops": 2.0 * n ** 3 / float(np.median(times[(n, kind)])) / 1e12} for n, kind in cases]


def run_one(M, N, K, variant, calls=5, alpha=1.0, beta=0.0, b_transposed=False):
    """A handful of calls of one shape with the default configuration, for profilers.
    variant: sgemm, f16tc (f32 operands), f16in (f16 operands, f32 C) or f16out (f16
    operands and C); b_transposed: B stored N x K."""
    import torch
    st = torch.cuda.current_stream().cuda_stream
    A = torch.rand(M, K, device="cuda") * 2 - 1
    B = torch.rand(K, N, device="cuda") * 2 - 1
    if b_transposed:
        B = B.t().contiguous()
    op_b = phx.OP_T if b_transposed else phx.OP_N
    C = torch.zeros(M, N, device="cuda")
    if variant in ("f16in", "f16out"):
        A, B = A.half(), B.half()
        if variant == "f16out":
            C = C.half()
        fn = phx.phx_gemm_f16in_f32acc if variant == "f16in" else phx.phx_gemm_f16in_f16out
        call = lambda: fn(0, op_b, M, N, K, alpha, A.data_ptr(), B.data_ptr(), beta, C.data_ptr(), st)
    else:
        fn = phx.phx_sgemm_ex if variant == "sgemm" else phx.phx_gemm_f16tc_f32acc_ex
        call = lambda: fn(0, op_b, M, N, K, alpha, A.data_ptr(), B.data_ptr(), beta, C.data_ptr(), st)
    for _ in range(calls):
        phx.check(call())
    torch.cuda.synchronize()
    return phx.get_config(0 if variant == "sgemm" else 1, M, N, K)


def main():
    ap = argparse.ArgumentParser(description="GEMM shape sweep on the roofline")
    ap.add_argument("--out", default=None)
    ap.add_argument("--quick", action="store_true", help="skip shapes above 2^40 MNK and shorten timings")
    ap.add_argument("--layouts", action="store_true", help="time the four storage orders at 4096^3 only")
    ap.add_argument("--skinny", action="store_true", help="time M = 1 .. 2048 rows against K = N = 4096 only")
    ap.add_argument("--narrow", action="store_true", help="time N = 1 .. 2048 columns against M = K = 4096 only")
    ap.add_argument("--b-transposed", action="store_true", help="with --skinny or --one: B stored N x K")
    ap.add_argument("--f16in", action="store_true", help="time half-precision operands against f32 ones only")
    ap.add_argument("--one", default=None, metavar="M,N,K", help="only run a few calls of this shape (for profilers)")
    ap.add_argument("--variant", default="sgemm", choices=("sgemm", "f16tc", "f16in", "f16out"), help="with --one")
    ap.add_argument("--calls", type=int, default=5, help="with --one")
    ap.add_argument("--alpha", type=float, default=1.0, help="with --one")
    ap.add_argument("--beta", type=float, default=0.0, help="with --one")
    args = ap.parse_args()
    if args.f16in:
        rows = run_f16in()
        for row in rows:
            print(f"{row['n']:6d}^3 {row['kind']:14s} {row['seconds'] * 1e6:9.1f} us {row['tflops']:8.1f} TFLOP/s")
        if args.out:
            with open(args.out, "w") as f:
                json.dump({"f16in": rows}, f, indent=1)
        return 0
    if args.one:
        M, N, K = (int(x) for x in args.one.split(","))
        print(f"{args.variant} {(M, N, K)} x{args.calls}: "
              f"{run_one(M, N, K, args.variant, args.calls, args.alpha, args.beta, args.b_transposed)}")
        return 0
    if args.skinny:
        rows = run_skinny(b_transposed=args.b_transposed)
        for row in rows:
            print(f"{row['variant']:6s} M={row['M']:5d} {row['seconds'] * 1e6:9.1f} us {row['tflops']:8.2f} TFLOP/s "
                  f"{row['gbs']:7.0f} GB/s  I={row['intensity']:7.1f}  [{row['config']}]")
        if args.out:
            with open(args.out, "w") as f:
                json.dump({"skinny": rows}, f, indent=1)
        return 0
    if args.narrow:
        rows = run_narrow()
        for row in rows:
            print(f"{row['variant']:6s} M={row['M']:5d} N={row['N']:5d} {row['seconds'] * 1e6:9.1f} us "
                  f"{row['tflops']:8.2f} TFLOP/s {row['gbs']:7.0f} GB/s  I={row['intensity']:7.1f}  [{row['config']}]")
        if args.out:
            with open(args.out, "w") as f:
                json.dump({"narrow": rows}, f, indent=1)
        return 0
    if args.layouts:
        rows = run_layouts()
        for row in rows:
            print(f"{row['variant']:6s} {row['layout']:>11s} {row['tflops']:8.1f} TFLOP/s  {row['vs_plain']:.3f}x of A @ B")
        if args.out:
            with open(args.out, "w") as f:
                json.dump({"layouts": rows}, f, indent=1)
        return 0
    res = run(quick=args.quick)
    r = res["roofs"]
    print(f"roofs: FP32 {r['fp32_ffma']['tflops']:.1f} / f32x2 {r['fp32_ffma2']['tflops']:.1f} TFLOP/s, "
          f"f16 tensor {r['f16_tensor']['tflops']:.0f} TFLOP/s, HBM read {r['hbm_read_gbs']:.0f} GB/s")
    for row in res["rows"]:
        print(f"{row['shape']:>16s} {row['variant']:6s} {row['tflops']:8.1f} TFLOP/s  "
              f"{row['pct_of_roof']:5.1f}% of {row['bound']} roof ({row['roof_tflops']:.0f})  "
              f"queued {row['queued_tflops']:8.1f} TFLOP/s  host {row['host_us_per_call']:5.1f} us/call  "
              f"[{row['config']}]")
    if args.out:
        with open(args.out, "w") as f:
            json.dump(res, f, indent=1)
    return 0


if __name__ == "__main__":
    sys.exit(main())
