"""The multi-rank path of bench.py on CPU: two gloo ranks, each timing its own replica of the
step, must agree on the slowest rank's time and report the whole job's throughput."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, ws, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    local_seconds = [1.5, 2.0][rank]          # rank 1 is the slower replica
    slowest = bench.reduce_max(local_seconds, ws)
    value = bench.whole_job_tflops(ws, steps=10, flops_per_step=3e12, max_seconds=slowest)
    q.put((rank, slowest, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in out:
        assert slowest == 2.0
        # 2 ranks x 10 steps x 3 TFLOP over the slowest rank's 2 s
        assert value == pytest.approx(2 * 10 * 3e12 / 2.0 / 1e12)


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(1.25, 1) == 1.25
    assert bench.whole_job_tflops(1, 4, 2e12, 0.5) == pytest.approx(16.0)


def _run_stub(argv, env_extra=None, drop_dist_env=True):
    import json
    import subprocess
    env = dict(os.environ)
    if drop_dist_env:
        for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
            env.pop(k, None)
    env.update(env_extra or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "bench_stub_rank.py"), *argv],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    return r, [json.loads(ln) for ln in lines]


def test_gpus_2_starts_two_ranks_and_reports_the_slowest():
    # bench.main with --gpus 2 and no outside launcher starts two ranks itself; each runs the
    # stand-in replica (rank r: steps of 1 + r ms) and rank 0 alone prints the line
    steps = 5
    r, lines = _run_stub(["--gpus", "2", "--steps", str(steps), "--warmup", "3", "--no-cpu-baseline"])
    assert r.returncode == 0, r.stderr[-3000:]
    assert len(lines) == 1, r.stdout
    out = lines[0]
    assert out["n_gpus"] == 2
    assert out["scaling"] == "weak"
    assert out["ms_per_step"] == pytest.approx(2.0)                 # the slower rank's step
    flops_per_step = 2 * 2.0 * 4096 ** 3
    assert out["value"] == pytest.approx(2 * steps * flops_per_step / (steps * 2e-3) / 1e12)
    # e2e: the slower rank's median run of 4 steps (4 x 2 x 2 ms), both ranks' work
    assert out["e2e"]["value"] == pytest.approx(2 * 4 * flops_per_step / 16e-3 / 1e12)
    assert out["config"]["parallelism"] == "replicas x2 (no collective)"


def test_rank_count_must_match_gpus():
    r, lines = _run_stub(["--gpus", "2", "--steps", "3", "--warmup", "3"],
                         env_extra={"WORLD_SIZE": "1", "RANK": "0", "LOCAL_RANK": "0"})
    assert r.returncode != 0
    assert not lines
    assert "WORLD_SIZE=1" in r.stderr
