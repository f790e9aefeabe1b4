"""The bounds-checked build (libshmm_checked.so, compiled with SHMM_CHECKED)
on the GPU: the parity and host-memory suites run again in a child process
with SHMM_CHECKED=1, so every global index their kernels compute is compared
with the extent of the buffer it addresses.  An index outside would skip the
access and leave SHMM_ERR_BOUNDS in the device status word, which every
test's status check then reports; a pass also shows that the checks change
no result."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gpu_suites_pass_under_bounds_checks():
    from partial_sum_reduction_gb300 import build
    build.build(checked=True)
    env = dict(os.environ, SHMM_CHECKED="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           os.path.join("tests", "test_gpu_parity.py"), os.path.join("tests", "test_gpu_host_run.py")]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0, r.stdout[-6000:] + r.stderr[-3000:]
    assert " passed" in r.stdout and "failed" not in r.stdout, r.stdout[-3000:]
