"""The C ABI used from plain C (tests/c/abi_smoke.c): compiled with gcc
against include/shmm.h and libshmm.so alone.  On the CPU it plans the
ownership page's worked example and checks the planner's answers and
errors; on a GPU it also runs an integer-valued sharded matmul through
shmm_run and shmm_run_host and compares every element with a host loop."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "partial_sum_reduction_gb300")
SRC = os.path.join(ROOT, "tests", "c", "abi_smoke.c")


def _cuda_root():
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path, gpu):
    if not shutil.which("gcc"):
        pytest.skip("gcc not available")
    from partial_sum_reduction_gb300 import build
    build.build()
    exe = str(tmp_path / ("abi_smoke_gpu" if gpu else "abi_smoke"))
    cmd = ["gcc", "-std=c11", "-O1", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), SRC,
           "-L", PKG, "-lshmm", "-Wl,-rpath," + PKG, "-o", exe]
    if gpu:
        cuda = _cuda_root()
        cmd[1:1] = ["-DSHMM_C_GPU", "-I", os.path.join(cuda, "include")]
        cmd += ["-L", os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(cuda, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_plans_the_worked_example(tmp_path):
    exe = _build(tmp_path, gpu=False)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "OK", r.stdout + r.stderr


@pytest.mark.gpu
def test_c_program_runs_the_sharded_matmul(tmp_path):
    exe = _build(tmp_path, gpu=True)
    r = subprocess.run([exe, "--gpu"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "OK", r.stdout + r.stderr
