"""bench.py's multi-process path on CPU with gloo, world size 2: the barrier
and max-over-ranks timing, and the reference arm under torchrun (rank 0
reports, the other rank exits 0 without work)."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "SHMM_BENCH_BACKEND": "gloo"})
    sys.path.insert(0, ROOT)
    import bench
    ctx = bench.DistCtx()
    ctx.barrier()
    m = ctx.max(10.0 * rank + 1.25)
    ctx.barrier()
    ctx.close()
    with open(os.path.join(out_dir, "r%d" % rank), "w") as f:
        f.write(repr(m))


def test_max_over_ranks_with_gloo(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    for r in range(2):
        assert float(open(tmp_path / ("r%d" % r)).read()) == 11.25


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    env = dict(os.environ, SHMM_BENCH_BACKEND="gloo", CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "down_projection_quarter", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--reference-budget-s", "4"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["value"] > 0 and out["unit"] == "TFLOP/s"
    assert out["n_gpus"] == 2 and out["e2e"]["h2d_bytes_per_step"] == 0
    assert out["cpu_baseline"]["kind"] == "oracle" and out["cpu_baseline"]["cores"] >= 1
