"""The bounds-checked build of libphx (PHX_DEBUG=1: every kernel checks its indices, tile
coordinates and tensor-memory columns, counting failures instead of trapping) runs the edge
sweep and every schedule's shapes with oracle-exact results and no failed check.

Built here on first use (nvcc, a minute or two), loaded in a child process through
PHX_LIBRARY so that this process keeps the normal build.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bounds_checked_build_runs_every_schedule_cleanly():
    sys.path.insert(0, ROOT)
    from dense_gemm_04_gb300 import build
    lib = build.build(debug=True)
    env = dict(os.environ, PHX_LIBRARY=lib)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "debug_sweep.py")], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert "violations 0" in r.stdout and "failures 0" in r.stdout, r.stdout


def test_normal_build_has_no_checks():
    sys.path.insert(0, ROOT)
    from dense_gemm_04_gb300 import phx
    assert phx.phx_debug_build() == 0
    assert phx.debug_violations() == 0
