"""GPU: the bounds-checked build keeps every kernel access inside its buffer.

No memory checker runs these tests, so the library is also built with ZERO_BOUNDS_CHECK:
each global access of the kernels' main paths is tested against the extent of the buffer
it belongs to, and the first access outside is recorded (and skipped). A child process
loads that build (ZERO_LIBZERO), runs every kernel of the step and the gather on workloads
that span many tiles, ragged tails, run-time rank counts and misaligned layouts, compares
each result with the oracle, and reads the bounds report, which must show no fault; then
the build's self-test shows that a range outside its buffer is recorded.
"""
import json
import os
import subprocess
import sys

import pytest

import sharded_emulated_reduce_gb300 as z

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_keeps_every_kernel_access_in_bounds():
    from sharded_emulated_reduce_gb300 import build
    path = build.build(checked=True)
    env = dict(os.environ, ZERO_LIBZERO=path)
    out = subprocess.run([sys.executable, os.path.join(HERE, "bounds_workloads.py")], env=env,
                         capture_output=True, text=True, timeout=1200)
    assert out.returncode == 0, out.stderr[-3000:]
    rep = json.loads(out.stdout.strip().splitlines()[-1])
    assert rep["enabled"] == 1, "the child did not load the checked build"
    assert rep["site"] == 0, rep
    assert all(rep["exact"].values()), rep["exact"]
    # and the checks do catch a range outside its buffer (the self-test's, never accessed)
    assert rep["probe"] == {"enabled": 1, "site": 11, "offset": 80}


def test_normal_build_reports_no_checks():
    z.zero_selftest_bounds()
    assert z.zero_bounds_check() == {"enabled": 0, "site": 0, "offset": 0}
