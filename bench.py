"""Benchmark of the GEMM hot path: C = alpha * A @ B + beta * C at M = N = K = 4096.

One step is one pass of the whole path on one batch of inputs: the f32 SIMT GEMM
(phx_sgemm) and the f16-tensor-core / f32-accumulate GEMM (phx_gemm_f16tc_f32acc, i.e.
its f32 -> f16 cast pass plus the tcgen05 GEMM), both with alpha = 1, beta = 0.5, on the
same synthetic A and B (uniform [-1, 1), splitmix64, seed 0) and each on its own C.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  `value` is the whole job's GEMM throughput, sum of 2MNK over the
GEMMs of all steps on all ranks divided by the slowest rank's summed device time of its
steps (CUDA events on the launching stream; L2 flushed between steps, outside the events).
`e2e` is the same metric through the public C ABI with host buffers: the pinned-host copies
of each step's inputs in, the GEMMs, and the results back out, all inside the timed region,
with the copies of neighbouring steps overlapping the GEMMs (two buffer sets, three streams);
`e2e.serial` runs the same steps one after another on one stream.
`roofline` places the dominant kernel (the f32 SIMT GEMM) against the FP32 issue rate of
the SMs; `roofline_tc_gemm` and `roofline_cast` place the tensor-core GEMM kernel and the
cast pass against the measured tensor and HBM peaks.  `cpu_baseline` times the CPU oracle
on a bounded sample of the same workload.

--impl reference times that oracle as the reference arm (there is no runnable reference
implementation: the pages describe their kernels but ship no library).

The path does not shard in this build, so with N GPUs each rank runs its own replica of
the step (no collective on the data path) and `scaling` is "weak".  `--gpus N` with N > 1,
run as a plain script, starts N ranks itself (torch.distributed.run, one process per GPU,
rank r on GPU r); under an outside torchrun launch WORLD_SIZE must equal N.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (2MNK/t) at M=N=K=4096, f32 SIMT & f16-TC/f32-acc; % of peak"
M = N = K = 4096
ALPHA, BETA = 1.0, 0.5
FLOPS_PER_GEMM = 2.0 * M * N * K
GEMMS_PER_STEP = 2
WORKLOAD = ("C = alpha*A@B + beta*C, M=N=K=4096, alpha=1, beta=0.5, row-major f32; "
            "one step = phx_sgemm (f32 SIMT) + phx_gemm_f16tc_f32acc (f16 tensor cores, f32 acc)")
DATA = "synthetic: A, B, C i.i.d. uniform[-1,1) f32 from splitmix64, seed 0 (no dataset involved)"
FP32_LANES_PER_SM = 128  # FP32 multiply-add lanes per SM on sm_100-family GPUs


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, ws: int, device=None) -> float:
    """The largest x over all ranks (the slowest rank's time); x itself on one rank."""
    if ws == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, ws: int, device=None) -> float:
    """The sum of x over all ranks; x itself on one rank."""
    if ws == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def whole_job_tflops(ws: int, steps: int, flops_per_step: float, max_seconds: float) -> float:
    """Throughput of the whole job: the work of every rank over the slowest rank's time.
    Each rank runs its own replica of the step (the path is not sharded), so the work grows
    with the number of ranks (weak scaling)."""
    return ws * steps * flops_per_step / max_seconds / 1e12


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "sm_max_mhz": float(p.get("sm_max_mhz", 2070.0)), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": 2070.0, "source": "fallback"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def f16_peak(peaks: dict, clocks: dict) -> tuple[float, str]:
    """Denominator of the tensor-core fractions: the measured burst bf16 rate (dense f16 runs
    at the bf16 rate), which applies to a kernel timed alone or in a short step at the
    maximum clock; scaled by the run's median SM clock when that was below the maximum or a
    throttle reason was active."""
    burst = peaks["bf16_tflops"]
    mhz, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz") or peaks["sm_max_mhz"]
    if mhz and (clocks.get("reasons") or mhz < 0.98 * mx):
        return burst * mhz / mx, f"{peaks['source']} bf16 burst x run clock {mhz:.0f}/{mx:.0f} MHz"
    return burst, f"{peaks['source']} bf16 burst (run at {mhz or mx:.0f} MHz, no throttle reason)"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._t.join(timeout=5)

    def summary(self):
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "power_w_max": max(pw),
                "reasons": sorted(reasons), "samples": len(sm)}


def _oracle_sample(seconds_target: float, max_rows: int | None = None):
    """Time the CPU oracle on leading row blocks of the workload (both variants) and return
    (TFLOP/s, rows used, seconds, threads).  The oracle is used exactly as it stands."""
    import oracle
    from dense_gemm_04_gb300 import synth
    oracle.build()
    B = synth.matrix(K, N, seed=0, tensor=synth.TENSOR_B)
    A_full = synth.matrix(M, K, seed=0, tensor=synth.TENSOR_A)
    C_full = synth.matrix(M, N, seed=0, tensor=synth.TENSOR_C)

    def run(rows):
        t0 = time.perf_counter()
        oracle.gemm(A_full[:rows], B, C_full[:rows], ALPHA, BETA, f16_inputs=False, want_mag=False)
        oracle.gemm(A_full[:rows], B, C_full[:rows], ALPHA, BETA, f16_inputs=True, want_mag=False)
        return time.perf_counter() - t0

    # per-row cost from two probes (each call also has a fixed cost: rounding B for the f16
    # variant), then one run sized to the target
    t32, t64 = run(32), run(64)
    per_row = max((t64 - t32) / 32, 1e-6)
    fixed = max(t32 - 32 * per_row, 0.0)
    rows = int((seconds_target - fixed) / per_row)
    rows = max(64, min(rows, max_rows or M, M))
    t = run(rows)
    flops = GEMMS_PER_STEP * 2.0 * rows * N * K
    return flops / t / 1e12, rows, t, oracle.num_threads()


def reference_arm(args):
    ws, rank, _ = _dist_env()
    if rank != 0:
        return 0
    import oracle
    from dense_gemm_04_gb300 import synth
    oracle.build()
    B = synth.matrix(K, N, seed=0, tensor=synth.TENSOR_B)
    A_full = synth.matrix(M, K, seed=0, tensor=synth.TENSOR_A)
    C_full = synth.matrix(M, N, seed=0, tensor=synth.TENSOR_C)
    rows = args.reference_rows

    def step():
        oracle.gemm(A_full[:rows], B, C_full[:rows], ALPHA, BETA, f16_inputs=False, want_mag=False)
        oracle.gemm(A_full[:rows], B, C_full[:rows], ALPHA, BETA, f16_inputs=True, want_mag=False)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    t = time.perf_counter() - t0
    flops = args.steps * GEMMS_PER_STEP * 2.0 * rows * N * K
    value = flops / t / 1e12
    sample = (f"each step: the oracle on the first {rows} of {M} rows of both GEMMs of the "
              f"workload ({rows}x{N}x{K}, f32 and f16-rounded inputs, float64 sums)")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
           "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": DATA,
           "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "alpha": ALPHA, "beta": BETA,
                      "reference": "CPU oracle (plain float64 triple loop, OpenMP over rows)"},
           "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return 0


KERNEL_SOURCES = {"sgemm": ("sgemm_simt.cu", "sgemm_tile_body.inc", "internal.h", "debug_checks.cuh"),
                  "tc_gemm": ("gemm_f16tc.cu", "sm100_ptx.cuh", "internal.h", "debug_checks.cuh"),
                  "f16_cast": ("gemm_f16tc.cu", "internal.h", "debug_checks.cuh")}


def kernel_source_hash(kernel: str) -> str:
    """sha256[:16] over the source files a kernel is compiled from, in a fixed order."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "dense_gemm_04_gb300", "csrc", name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def _traffic_from_profiles(kernel: str):
    """DRAM bytes per call recorded from ncu captures, if none of the kernel's source files has
    changed since (profiles/dram_traffic.txt: kernel, bytes per call, hash of its sources; a
    call of the f32 GEMM at 4096^3 is three kernels, summed there)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    h = kernel_source_hash(kernel)
    with open(path) as f:
        for line in f:
            p = line.split()
            if len(p) >= 3 and not line.startswith("#") and p[0] == kernel and p[2] == h:
                return float(p[1])
    return None


def measure_replica(args, local: int, ws: int) -> dict:
    """Time this rank's replica of the step on GPU `local`; returns its raw measurements."""
    import torch
    import torch.distributed as dist
    from dense_gemm_04_gb300 import phx, synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    props = torch.cuda.get_device_properties(local)

    # inputs resident in HBM before any timing
    hA = synth.matrix(M, K, seed=0, tensor=synth.TENSOR_A)
    hB = synth.matrix(K, N, seed=0, tensor=synth.TENSOR_B)
    hC = synth.matrix(M, N, seed=0, tensor=synth.TENSOR_C)
    A = torch.from_numpy(hA).to(dev)
    B = torch.from_numpy(hB).to(dev)
    C32 = torch.from_numpy(hC).to(dev)
    C16 = C32.clone()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)   # > 129 MB L2

    def sgemm():
        phx.check(phx.phx_sgemm(M, N, K, ALPHA, A.data_ptr(), B.data_ptr(), BETA, C32.data_ptr(), sh))

    def f16():
        phx.check(phx.phx_gemm_f16tc_f32acc(M, N, K, ALPHA, A.data_ptr(), B.data_ptr(), BETA,
                                            C16.data_ptr(), sh))

    # settle the clocks under the same work, then the W warm-up steps (all untimed)
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < args.settle_s:
        sgemm()
        f16()
        torch.cuda.synchronize()
    for _ in range(args.warmup):
        sgemm()
        f16()
    torch.cuda.synchronize()

    # three events per step: start, between the two GEMM calls, end
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)                   # evict L2 (outside the step's events)
            ev[i][0].record(stream)
            sgemm()
            ev[i][1].record(stream)
            f16()
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    if ws > 1:
        dist.barrier()
    step_ms = [a.elapsed_time(c) for a, _, c in ev]
    sgemm_ms = [a.elapsed_time(b) for a, b, _ in ev]
    f16_ms = [b.elapsed_time(c) for _, b, c in ev]

    # Per-kernel device times, from a separate pass with the library's event profile on.
    # Events between the cast and the tensor-core GEMM serialise the two, so this pass times
    # each kernel alone; the timed steps above run them as the call does.
    prof_steps = max(10, min(args.steps, 50))
    phx.profile_start()
    for i in range(prof_steps):
        flush.fill_(i & 0xFF)
        sgemm()
        f16()
    torch.cuda.synchronize()
    prof = phx.profile_stop()
    st = phx.check_device_status()
    if st != phx.PHX_OK:
        raise RuntimeError(f"device status after the timed steps: {phx.status_string(st)}")

    # End to end through the public C ABI with host buffers: every step copies its inputs in
    # from pinned host memory and its two results back out, inside the timed region.  The
    # steps run the way a serving loop runs them: two buffer sets and three streams, so the
    # copies in of step i+1 and out of step i-1 overlap the GEMMs of step i.  The same steps
    # one after another on one stream are reported beside it ("serial").
    pA, pB = torch.from_numpy(hA).pin_memory(), torch.from_numpy(hB).pin_memory()
    pC = torch.from_numpy(hC).pin_memory()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bufs = []
    for _ in range(2):
        bufs.append({"A": torch.empty_like(A), "B": torch.empty_like(B), "C32": torch.empty_like(C32),
                     "C16": torch.empty_like(C32), "o32": torch.empty_like(pC).pin_memory(),
                     "o16": torch.empty_like(pC).pin_memory(), "in": torch.cuda.Event(),
                     "comp": torch.cuda.Event(), "out": torch.cuda.Event()})

    def gemms(b):
        phx.check(phx.phx_sgemm(M, N, K, ALPHA, b["A"].data_ptr(), b["B"].data_ptr(), BETA, b["C32"].data_ptr(), sh))
        phx.check(phx.phx_gemm_f16tc_f32acc(M, N, K, ALPHA, b["A"].data_ptr(), b["B"].data_ptr(), BETA,
                                            b["C16"].data_ptr(), sh))

    def copy_in(b):
        b["A"].copy_(pA, non_blocking=True)
        b["B"].copy_(pB, non_blocking=True)
        b["C32"].copy_(pC, non_blocking=True)
        b["C16"].copy_(pC, non_blocking=True)

    def copy_out(b):
        b["o32"].copy_(b["C32"], non_blocking=True)
        b["o16"].copy_(b["C16"], non_blocking=True)

    def e2e_pipelined(nsteps):
        for i in range(nsteps):
            b = bufs[i % 2]
            with torch.cuda.stream(s_in):
                s_in.wait_event(b["comp"])   # the buffer's last GEMMs are done with it
                s_in.wait_event(b["out"])    # and its last results are out
                copy_in(b)
                b["in"].record(s_in)
            stream.wait_event(b["in"])
            gemms(b)
            b["comp"].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(b["comp"])
                copy_out(b)
                b["out"].record(s_out)

    def e2e_serial(nsteps):
        b = bufs[0]
        for _ in range(nsteps):
            copy_in(b)
            gemms(b)
            copy_out(b)

    # three timed runs of e2e_steps steps each; the median run is reported (the host's
    # memory system is shared with other work on the machine).  A run starts with one step's
    # copies in and ends with one step's copies out that nothing overlaps, so it takes 30 steps
    # to make that ramp small.
    e2e_steps = max(4, min(args.steps, 30))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_pipelined(2)
    torch.cuda.synchronize()
    runs = []
    for _ in range(3):
        e0.record(s_in)
        e2e_pipelined(e2e_steps)
        e1.record(s_out)
        torch.cuda.synchronize()
        runs.append(e0.elapsed_time(e1) / 1e3)
    serial_runs = []
    with torch.cuda.stream(stream):
        e2e_serial(2)
        torch.cuda.synchronize()
        for _ in range(3):
            e0.record(stream)
            e2e_serial(e2e_steps)
            e1.record(stream)
            torch.cuda.synchronize()
            serial_runs.append(e0.elapsed_time(e1) / 1e3)
    return {
        "sms": props.multi_processor_count, "step_ms": step_ms, "sgemm_ms": sgemm_ms, "f16_ms": f16_ms,
        "prof": prof, "prof_steps": prof_steps, "clocks": clk.summary(), "wall": wall,
        "e2e_steps": e2e_steps, "e2e_runs": runs, "e2e_serial_runs": serial_runs,
        "h2d": M * K * 4 + K * N * 4 + 2 * M * N * 4, "d2h": 2 * M * N * 4,
        "configs": {"sgemm": phx.get_config(0, M, N, K), "f16tc_f32acc": phx.get_config(1, M, N, K)},
    }


def gpu_arm(args, replica=None, backend=None):
    """One rank of the bench: time this rank's replica (measure_replica, or `replica` with the
    same signature), take the slowest rank's times, and print the JSON line on rank 0.  The
    process group is NCCL on GPUs (gloo without one, or as `backend` says); it carries only
    the barriers and the reductions of the timings."""
    import torch
    import torch.distributed as dist

    ws, rank, local = _dist_env()
    if ws != args.gpus:
        raise SystemExit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={ws}: one rank per GPU is required")
    backend = backend or ("nccl" if torch.cuda.is_available() else "gloo")
    if ws > 1:
        dist.init_process_group(backend)
    dev = torch.device("cuda", local) if backend == "nccl" else None
    peaks = _peaks()
    r = (replica or measure_replica)(args, local, ws)
    max_s = reduce_max(sum(r["step_ms"]) / 1e3, ws, dev)
    e2e_max_s = reduce_max(statistics.median(r["e2e_runs"]), ws, dev)
    serial_max_s = reduce_max(statistics.median(r["e2e_serial_runs"]), ws, dev)
    # every rank counts itself in: the line's n_gpus is the number of replicas that ran
    n_ranks = int(round(reduce_sum(1.0, ws, dev)))
    if n_ranks != args.gpus:
        raise SystemExit(f"bench.py: {n_ranks} ranks reported for --gpus {args.gpus}")
    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return 0

    value = whole_job_tflops(ws, args.steps, GEMMS_PER_STEP * FLOPS_PER_GEMM, max_s)
    clocks = r["clocks"]
    sms = r["sms"]
    sm_max = clocks.get("sm_max_mhz") or peaks["sm_max_mhz"]
    prof, prof_steps = r["prof"], r["prof_steps"]
    launches_per_step = sum(n for n, _ in prof.values()) / prof_steps
    launches = int(round(launches_per_step * args.steps))

    def per_call_ms(kind):
        # one call of each kind per step (a call may launch several kernels of its kind)
        n, ms = prof[kind]
        return ms / prof_steps if n else None

    sg_ms = per_call_ms("sgemm")
    tc_ms = per_call_ms("tc_gemm")
    cast_ms = per_call_ms("f16_cast")
    fp32_peak = sms * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
    run_mhz = clocks.get("sm_mhz")
    sg_tflops = FLOPS_PER_GEMM / (sg_ms / 1e3) / 1e12
    roofline = {"bound": "alu", "kernel": "sgemm (f32 SIMT, FFMA)", "achieved": sg_tflops,
                "peak": fp32_peak, "unit": "TFLOP/s", "frac": sg_tflops / fp32_peak,
                "traffic": _traffic_from_profiles("sgemm"),
                "peak_source": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 FLOP x {sm_max:.0f} MHz (max SM clock)",
                "algorithmic_bytes": 4.0 * (M * K + K * N + 2 * M * N)}
    if run_mhz:
        roofline["frac_at_run_clock"] = sg_tflops / (sms * FP32_LANES_PER_SM * 2 * run_mhz * 1e6 / 1e12)
    # the f16 call as it runs inside the timed steps (cast and GEMM as the call launches them)
    f16_call_ms = statistics.median(r["f16_ms"])
    f16_call_tflops = FLOPS_PER_GEMM / (f16_call_ms / 1e3) / 1e12
    tc_tflops = FLOPS_PER_GEMM / (tc_ms / 1e3) / 1e12
    tc_peak, tc_peak_src = f16_peak(peaks, clocks)
    roofline_tc = {"bound": "tensor", "kernel": "tcgen05 f16 GEMM (f32 accumulate), timed alone",
                   "achieved": tc_tflops, "peak": tc_peak, "unit": "TFLOP/s", "frac": tc_tflops / tc_peak,
                   "traffic": _traffic_from_profiles("tc_gemm"), "peak_source": tc_peak_src,
                   "algorithmic_bytes": 2.0 * (M * K + K * N) + 4.0 * 2 * M * N,
                   "call_tflops": f16_call_tflops, "call_frac": f16_call_tflops / tc_peak,
                   "call": "the whole phx_gemm_f16tc_f32acc call (cast + GEMM) in the timed steps"}
    cast_bytes = 6.0 * (M * K + K * N)
    cast_gbs = cast_bytes / (cast_ms / 1e3) / 1e9
    roofline_cast = {"bound": "hbm", "kernel": "f32->f16 cast pass (A and B, one launch), timed alone",
                     "achieved": cast_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": cast_gbs / peaks["hbm_gbs"], "traffic": _traffic_from_profiles("f16_cast"),
                     "algorithmic_bytes": cast_bytes}
    sg_call_ms = statistics.median(r["sgemm_ms"])
    variants = {
        "sgemm": {"tflops": FLOPS_PER_GEMM / (sg_call_ms / 1e3) / 1e12, "ms": sg_call_ms,
                  "kernels_alone_ms": sg_ms, "config": r["configs"]["sgemm"]},
        "f16tc_f32acc": {"tflops": f16_call_tflops, "ms": f16_call_ms, "gemm_kernel_alone_ms": tc_ms,
                         "cast_alone_ms": cast_ms, "frac_of_tensor_peak": f16_call_tflops / tc_peak,
                         "config": r["configs"]["f16tc_f32acc"]},
    }
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        v, rows, t, cores = _oracle_sample(args.cpu_seconds)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "cpu_model": cpu_model(), "kind": "oracle",
               "sample": f"the oracle on the first {rows} of {M} rows of both GEMMs of the workload "
                         f"({rows}x{N}x{K} each, f32 and f16-rounded inputs), {t:.1f} s"}
    e2e_steps = r["e2e_steps"]
    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": n_ranks, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * max_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 (SIMT) + f16xf16->f32 (tensor cores)",
        "data": DATA,
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "alpha": ALPHA, "beta": BETA,
                   "l2": "flushed between steps by a 512 MiB write outside the step's events",
                   "settle_s": args.settle_s, "parallelism": f"replicas x{ws} (no collective)"},
        "variants": variants,
        "roofline": roofline,
        "roofline_tc_gemm": roofline_tc,
        "roofline_cast": roofline_cast,
        "cpu_baseline": cpu,
        "e2e": {"value": whole_job_tflops(ws, e2e_steps, GEMMS_PER_STEP * FLOPS_PER_GEMM, e2e_max_s),
                "unit": "TFLOP/s", "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "steps": e2e_steps, "runs": len(r["e2e_runs"]), "run_ms": [1e3 * x for x in r["e2e_runs"]],
                "schedule": "copies in of step i+1 and out of step i-1 overlap the GEMMs of step i "
                            "(two buffer sets, three streams)",
                "serial": whole_job_tflops(ws, e2e_steps, GEMMS_PER_STEP * FLOPS_PER_GEMM, serial_max_s)},
        "clocks": clocks,
        "gpu_launches": launches,
        "kernel_launches_per_step": {k: v[0] / prof_steps for k, v in prof.items()},
        "kernel_times_from": f"a separate pass of {prof_steps} steps with per-kernel events",
        "wall_s_timed_region": r["wall"],
        "peaks": peaks,
    }
    print(json.dumps(out), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def launch_ranks(n: int, argv: list[str]) -> int:
    """Start n ranks of this script on this node (torch.distributed.run, one process per
    GPU, rendezvous on 127.0.0.1) and return the launcher's exit status."""
    import socket
    sock = socket.socket()
    sock.bind(("127.0.0.1", 0))
    port = sock.getsockname()[1]
    sock.close()
    script = os.path.abspath(sys.argv[0]) if sys.argv and sys.argv[0].endswith(".py") else os.path.abspath(__file__)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), script, *argv]
    return subprocess.call(cmd)


def main(argv=None, replica=None, backend=None):
    """Parse the command line and run one arm; with --gpus N > 1 outside a torchrun launch,
    start N ranks of the running script first.  `replica` and `backend` go to gpu_arm."""
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["phx", "reference"], default="phx")
    ap.add_argument("--settle-s", type=float, default=1.0, help="untimed settle time before warm-up")
    ap.add_argument("--cpu-seconds", type=float, default=8.0, help="target CPU seconds of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reference-rows", type=int, default=64,
                    help="rows of the workload the reference arm's oracle evaluates per step")
    args = ap.parse_args(argv)
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return launch_ranks(args.gpus, sys.argv[1:] if argv is None else list(argv))
    if args.impl == "reference":
        return reference_arm(args)
    return gpu_arm(args, replica=replica, backend=backend)


if __name__ == "__main__":
    sys.exit(main())
