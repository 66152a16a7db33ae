"""Runs bench.py's rank handling and aggregation with a CPU stand-in for the GPU replica
(the measurements a replica returns), over gloo, for tests/test_bench_multirank.py.

Rank r's stand-in replica reports steps of 1 + r milliseconds, so the slowest rank is the
last one.  `python tests/bench_stub_rank.py --gpus 2 ...` starts the ranks itself, as
`python bench.py --gpus 2 ...` does.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def stub_replica(args, local, ws):
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", "0"))
    ms = 1.0 + rank
    if ws > 1:
        dist.barrier()
    half = [ms / 2] * args.steps
    return {
        "sms": 152, "step_ms": [ms] * args.steps, "sgemm_ms": half, "f16_ms": half,
        "prof": {"sgemm": (3 * 10, 10 * ms / 2), "f16_cast": (10, 10 * ms / 8), "tc_gemm": (10, 10 * 3 * ms / 8),
                 "scale_c": (0, 0.0), "transpose": (0, 0.0), "skinny": (0, 0.0)},
        "prof_steps": 10,
        "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 0},
        "wall": args.steps * ms / 1e3, "e2e_steps": 4, "e2e_runs": [4 * 2 * ms / 1e3] * 3,
        "e2e_serial_runs": [4 * 3 * ms / 1e3] * 3, "h2d": 1, "d2h": 1,
        "configs": {"sgemm": "stub", "f16tc_f32acc": "stub"},
    }


if __name__ == "__main__":
    sys.exit(bench.main(replica=stub_replica, backend="gloo"))
