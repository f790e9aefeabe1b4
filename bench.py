#!/usr/bin/env python
"""Throughput of the sharded matmul hot path on GB300.

Default workload: the tensor-parallel down-projection of "Sharded matmuls and
collectives on a torus" (the sharding sandbox's default case 3): A[8192,28672]
. B[28672,8192] bf16 on mesh {X:4,Y:2}, A[I_X,J_Y], B[J_Y,K], result C[I_X,K]
(all-reduce over Y), entries N(0,1)/sqrt(28672).  Each of the 8 virtual ranks
multiplies a [2048,14336].[14336,8192] shard (481 GFLOP) and the partial sums
are reduced in the GEMM epilogue.  One step = one shmm_run over the whole
mesh (plan built once, outside the timed region).

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl shmm|reference]
        [--workload down_projection|four_case|mlp_pair|split_k_integer]
        python bench.py --sweep collectives     (reduce-scatter / all-reduce /
                                                 all-gather bandwidth sweep)
        python bench.py --sweep gemm            (the local GEMM beside cuBLAS)
Under torchrun (N > 1) every GPU runs its own replica of the workload (the
virtual-rank mesh lives on one GPU); the reported value is the work of all
replicas over the slowest replica's time (weak scaling).

Prints one JSON line (rank 0).
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("sharded-matmul TFLOP/s (% bf16 peak) and reduce-scatter GB/s (% HBM) on 1 GB300")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# device-side delay (SM cycles, ~0.1 ms) enqueued before a timed collective
SLEEP_CYCLES = 200000
L2_BYTES = 129 << 20
# datasheet figures of one GB300, reported beside the measured denominators
NOMINAL_PEAKS = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0}

WORKLOADS = {
    "down_projection": dict(
        mesh=[("X", 4), ("Y", 2)], sA=(("X",), ("Y",)), sB=(("Y",), ()), sC=(("X",), ()),
        I=8192, J=28672, K=8192, fused=True,
        text="tensor-parallel down-projection A[8192,28672].B[28672,8192] bf16 on {X:4,Y:2}, "
             "A[I_X,J_Y], B[J_Y,K] -> C[I_X,K] (all-reduce over Y fused into the GEMM epilogue)"),
    "down_projection_quarter": dict(
        mesh=[("X", 4), ("Y", 2)], sA=(("X",), ("Y",)), sB=(("Y",), ()), sC=(("X",), ()),
        I=4096, J=14336, K=4096, fused=True,
        text="quarter-size down-projection A[4096,14336].B[14336,4096] bf16 on {X:4,Y:2} (profiling case)"),
    "four_case": dict(
        mesh=[("X", 2), ("Y", 2)], I=2048, J=2048, K=2048, fused=True,
        text="four-case sweep I=J=K=2048 bf16 on {X:2,Y:2} (cases 1-4 back to back)"),
    "mlp_pair": dict(
        mesh=[("X", 8)], T=8192, D=4096, F=16384, fused=True,
        text="MLP column->row pair X[8192,4096].W1[4096,16384] (GeLU) .W2[16384,4096] bf16 on {X:8}, "
             "all-reduce of Y fused"),
    "mlp_pair_sp": dict(
        mesh=[("X", 8)], T=8192, D=4096, F=16384, fused=True,
        text="sequence-parallel MLP block on {X:8}: X[8192,4096].W1 (GeLU) .W2 reduce-scattered over "
             "tokens (fused), then LayerNorm per token fused with the all-gather"),
    "split_k_integer": dict(
        mesh=[("Y", 2)], I=64, J=64, K=64, fused=True,
        text="split-K integer fp32 A[64,64].B[64,64] on {Y:2}, reduce-scatter C[I_Y,K]"),
}
FOUR_CASES = [
    ((("X",), ()), ((), ("Y",)), (("X",), ("Y",))),
    (((), ("X",)), ((), ()), ((), ())),
    (((), ("Y",)), (("Y",), ()), (("Y",), ())),
    ((("X",), ()), ((), ("X",)), (("X",), ())),
]


# DRAM bytes per launch of the dominant kernel from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum, one pass, full-size launch:
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none
#       -k regex:gemm_tc2 -s 3 -c 1 python bench.py --steps 5 --warmup 3 --no-cpu-baseline),
# valid only for the kernel code it was taken on (kernel_source_hash).
NCU_TRAFFIC = {
    "down_projection": {"kernel_sha256_16": "18b29c5ca3e12890", "bytes": 4.131820032e9 + 0.246573312e9,
                        "kernel": "gemm_tc2_kernel<2> (256x512 tiles)",
                        "note": ("one capture on the current source (4.13 GB read + 0.25 GB written at "
                                 "1.95 ms); the same tile schedule has read 3.08-3.70 GB on most boxes and "
                                 "4.13-5.94 GB on others, against a wave model of 3.35 GB and 2.62 GB "
                                 "algorithmic")},
}


def kernel_source_hash():
    """sha256 (16 hex digits) of the GEMM kernel's source with comments and
    blank space removed, so a comment edit keeps a capture valid while any
    change to the code voids it."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in ("gemm_tcgen05.cu", "device_wait.cuh", "checked.cuh", "gelu.cuh"):
        with open(os.path.join(ROOT, "partial_sum_reduction_gb300", "csrc", name)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def kernel_traffic(workload):
    rec = NCU_TRAFFIC.get(workload)
    if not rec:
        return None
    return rec["bytes"] if kernel_source_hash() == rec["kernel_sha256_16"] else None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"]))}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of the SM clock and throttle reasons; only samples
    stamped inside [mark_start, mark_end] count."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, bus_id=None, interval_ms=50):
        self.proc = None
        self.t_start = self.t_end = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
               "-lms", str(interval_ms)]
        if bus_id:
            cmd += ["-i", bus_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    @staticmethod
    def _ts(text):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(text.strip(), fmt).timestamp()
            except ValueError:
                pass
        return None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        rows = []
        for line in self.out.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((self._ts(parts[0]), float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.out.name)
        inside = [r for r in rows if r[0] is not None and self.t_start is not None and
                  self.t_start - 0.05 <= r[0] <= self.t_end + 0.05]
        window = "timed region"
        if not inside:
            inside, window = rows, "whole run (no sample fell inside the timed region)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        reasons = sorted({self.NAMES[i] for r in inside for i, f in enumerate(r[3]) if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


# ------------------------------------------------------------- workloads

class Workload:
    """Plans, per-rank device buffers and pinned host copies of one workload;
    ``step()`` enqueues one pass of the hot path."""

    def __init__(self, name, device, rank_order=False, sm_split=True, batch=True):
        import torch
        import partial_sum_reduction_gb300 as s
        import shmm_inputs
        from partial_sum_reduction_gb300 import helpers as H
        self.name, self.cfg = name, WORKLOADS[name]
        self.s, self.H, self.torch = s, H, torch
        c = self.cfg
        self.steps_spec = []   # (plan, A list, B list, C list, ws)
        self.flops = 0
        FUSED = s.FLAG_FUSED | (s.FLAG_RANK_ORDER if rank_order else 0)
        if name in ("down_projection", "down_projection_quarter"):
            A, B = shmm_inputs.scaled_normal_pair(c["I"], c["J"], c["K"], "bf16", seed=0)
            self.host_globals = (A, B)
            self._add(c["mesh"], c["sA"], c["sB"], c["sC"], A, B, FUSED if c["fused"] else 0, device)
        elif name == "four_case":
            A, B = shmm_inputs.scaled_normal_pair(c["I"], c["J"], c["K"], "bf16", seed=0)
            self.host_globals = (A, B)
            for sA, sB, sC in FOUR_CASES:
                self._add(c["mesh"], sA, sB, sC, A, B, FUSED, device)
            # The four cases are independent.  Each alone is 1-2 waves of
            # tiles and would take every SM with a partial last wave.  By
            # default one shmm_run_batch call runs their GEMMs as one launch
            # (one tile walk over all four); otherwise they run on their own
            # streams with the GPU split among them by their share of the
            # FLOPs (whole CTA pairs, at least one each).
            self.batch = batch
            self.sm_split = None
            if sm_split and not batch:
                sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
                fl = [p.info.flops_per_rank * p.nranks for p, *_ in self.steps_spec]
                pairs = [max(1, int(round(sms // 2 * f / sum(fl)))) for f in fl]
                while sum(pairs) > sms // 2:
                    pairs[pairs.index(max(pairs))] -= 1
                self.sm_split = [2 * n for n in pairs]
                for (p, *_), n in zip(self.steps_spec, self.sm_split):
                    p.set_sm_limit(n)
        elif name == "mlp_pair":
            X, W1, W2 = shmm_inputs.mlp_pair(c["T"], c["D"], c["F"], seed=0)
            self.host_globals = (X, W1, W2)
            p1 = self._add(c["mesh"], ((), ()), ((), ("X",)), ((), ("X",)), X, W1, s.FLAG_GELU, device)
            H_r = self.steps_spec[0][3]
            p2 = s.Plan(c["mesh"], ((), ("X",)), (("X",), ()), ((), ()), c["T"], c["F"], c["D"], "bf16", "bf16",
                        FUSED)
            W2_r = H.shard(p2, s.TENSOR_B, W2, device)
            Y_r = H.alloc(p2, s.TENSOR_C, device)
            self.steps_spec.append((p2, H_r, W2_r, Y_r, H.workspace(p2, device)))
            self.flops += p2.info.flops_per_rank * p2.nranks
        elif name == "mlp_pair_sp":
            X, W1, W2 = shmm_inputs.mlp_pair(c["T"], c["D"], c["F"], seed=0)
            self.host_globals = (X, W1, W2)
            self._add(c["mesh"], ((), ()), ((), ("X",)), ((), ("X",)), X, W1, s.FLAG_GELU, device)
            H_r = self.steps_spec[0][3]
            p2 = s.Plan(c["mesh"], ((), ("X",)), (("X",), ()), (("X",), ()), c["T"], c["F"], c["D"], "bf16",
                        "bf16", FUSED)
            W2_r = H.shard(p2, s.TENSOR_B, W2, device)
            Y_r = H.alloc(p2, s.TENSOR_C, device)
            self.steps_spec.append((p2, H_r, W2_r, Y_r, H.workspace(p2, device)))
            self.flops += p2.info.flops_per_rank * p2.nranks
            self.sp_gather = s.Plan(c["mesh"], (("X",), ()), ((), ()), ((), ()), c["T"], 8, c["D"], "bf16", "bf16")
            self.sp_out = H.alloc(self.sp_gather, s.TENSOR_C, device)
            self.sp_gamma = torch.ones(c["D"], dtype=torch.float32, device=device)
            self.sp_beta = torch.zeros(c["D"], dtype=torch.float32, device=device)
        elif name == "split_k_integer":
            A, B = shmm_inputs.split_k_integer(c["I"], c["J"], c["K"], seed=0)
            self.host_globals = (A, B)
            self._add(c["mesh"], ((), ("Y",)), (("Y",), ()), (("Y",), ()), A, B, FUSED, device,
                      dt="f32")
        torch.cuda.synchronize()

    def _add(self, mesh, sA, sB, sC, A, B, flags, device, dt="bf16"):
        s, H = self.s, self.H
        I, J = A.shape
        K = B.shape[1]
        p = s.Plan(mesh, sA, sB, sC, I, J, K, dt, dt, flags)
        A_r, B_r = H.shard(p, s.TENSOR_A, A, device), H.shard(p, s.TENSOR_B, B, device)
        C_r = H.alloc(p, s.TENSOR_C, device)
        self.steps_spec.append((p, A_r, B_r, C_r, H.workspace(p, device)))
        self.flops += p.info.flops_per_rank * p.nranks
        return p

    def step(self, stream):
        if self.name == "four_case" and self.batch:
            sp = self.steps_spec
            self.s.shmm_run_batch([x[0] for x in sp], [x[1] for x in sp], [x[2] for x in sp], [x[3] for x in sp],
                                  [x[4] for x in sp], stream=stream)
            return
        if self.name == "four_case":
            # four independent sharded matmuls: forked onto their own streams
            # so one case's last partial wave overlaps the next case's work
            torch = self.torch
            if not hasattr(self, "side"):
                self.side = [torch.cuda.Stream() for _ in self.steps_spec[1:]]
            for st in self.side:
                st.wait_stream(stream)
            for i, (p, A_r, B_r, C_r, ws) in enumerate(self.steps_spec):
                st = stream if i == 0 else self.side[i - 1]
                p.run(A_r, B_r, C_r, ws, stream=st)
            for st in self.side:
                stream.wait_stream(st)
            return
        for p, A_r, B_r, C_r, ws in self.steps_spec:
            p.run(A_r, B_r, C_r, ws, stream=stream)
        if self.name == "mlp_pair_sp":
            self.sp_gather.layernorm_all_gather(self.steps_spec[-1][3], self.sp_gamma, self.sp_beta, self.sp_out,
                                                stream=stream)

    def input_bytes(self):
        n = 0
        for i, (p, A_r, B_r, C_r, ws) in enumerate(self.steps_spec):
            if self.name in ("mlp_pair", "mlp_pair_sp") and i == 1:
                n += sum(t.numel() * t.element_size() for t in B_r)
                continue
            n += sum(t.numel() * t.element_size() for t in A_r + B_r)
        return n

    def output_tensors(self):
        if self.name == "mlp_pair":
            return self.steps_spec[-1][3]
        if self.name == "mlp_pair_sp":
            return self.sp_out
        out = []
        for p, A_r, B_r, C_r, ws in self.steps_spec:
            out += C_r
        return out


def capture_graph(wl):
    """One step of the hot path captured into a CUDA graph (the plan's
    kernels with their arguments); replaying it removes the host-side
    marshalling and launch cost that dominates steps of a few microseconds."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            wl.step(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        wl.step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    return g


def time_device(wl, steps, warmup, dist_ctx, graph=False):
    """Device-timed loops on the launching stream; inputs (>> L2 for the
    full-size workloads) stay resident.  The timed region is `steps` steps
    back to back between two CUDA events, with nothing else in the stream:
    the total, the launch count and the clocks come from it.  The same
    number of steps then runs again, each between its own pair of events,
    for the per-step durations (median, best, and the roofline's launch
    duration).  An event between two launches keeps the later one from
    starting before the earlier has ended, which costs a few per cent on
    0.1 ms steps."""
    import torch
    s = wl.s
    stream = torch.cuda.current_stream()
    step = (lambda st: g.replay()) if graph else wl.step
    if graph:
        g = capture_graph(wl)
        launches_per_step = s.shmm_kernel_launches()
        wl.step(stream)  # count one step's kernels (a replay does not call the library)
        torch.cuda.synchronize()
        launches_per_step = s.shmm_kernel_launches() - launches_per_step
    for _ in range(warmup):
        step(stream)
    torch.cuda.synchronize()
    s.shmm_sync_status(stream)
    dist_ctx.barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    bus = None
    try:
        bus = torch.cuda.get_device_properties(torch.cuda.current_device()).pci_bus_id
    except Exception:
        pass
    sampler = ClockSampler(bus_id=_smi_bus_id(bus))
    time.sleep(0.3)
    launches0 = s.shmm_kernel_launches()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    sampler.mark_start()
    t0.record(stream)
    for i in range(steps):
        step(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    sampler.mark_end()
    launches = s.shmm_kernel_launches() - launches0
    if graph:
        launches = launches_per_step * steps
    clocks = sampler.stop()
    s.shmm_sync_status(stream)
    total_ms = t0.elapsed_time(t1)
    for i in range(steps):
        ev[i][0].record(stream)
        step(stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    s.shmm_sync_status(stream)
    per_step = [a.elapsed_time(b) for a, b in ev]
    total_ms = dist_ctx.max(total_ms)
    return total_ms, per_step, launches, clocks


def _smi_bus_id(bus):
    if not bus:
        return None
    # torch reports e.g. "0000:1B:00.0"; nvidia-smi accepts "00000000:1B:00.0"
    parts = bus.split(":")
    if len(parts) == 3 and len(parts[0]) == 4:
        return "0000" + bus
    return bus


def _distinct_bytes(plan, tensor, elem):
    """Bytes of the distinct boxes of ``tensor`` over the ranks (replicas
    counted once): what crosses the host link for it."""
    seen = {}
    for r in range(plan.nranks):
        off, ext = plan.rank_box(tensor, r)
        seen[tuple(off)] = ext[0] * ext[1] * elem
    return sum(seen.values())


def time_e2e(wl, steps, dist_ctx, windows=5):
    """End to end through the public API from host memory: every step
    uploads the global operands from pinned host memory (shmm_run_host:
    each distinct shard once, replicas copied on the device, uploads of one
    reduction group overlapping the previous group's GEMM), runs the sharded
    matmul, and writes the global result back to pinned host memory, all
    inside the timed region.  Chained steps keep their intermediate on the
    device (a NULL host operand)."""
    import torch
    s = wl.s
    stream = torch.cuda.current_stream()
    pin = lambda t: t.pin_memory()
    calls = []          # (plan, A_host|None, B_host|None, C_host|None, A_r, B_r, C_r, ws)
    h2d = d2h = 0
    final_copy = None
    specs = wl.steps_spec
    if wl.name in ("mlp_pair", "mlp_pair_sp"):
        X, W1, W2 = (pin(t) for t in wl.host_globals)
        (p1, X_r, W1_r, H_r, ws1), (p2, _, W2_r, Y_r, ws2) = specs
        last_out = None
        if wl.name == "mlp_pair":
            last_out = torch.empty(p2.shape[0], p2.shape[2], dtype=torch.bfloat16).pin_memory()
        calls.append((p1, X, W1, None, X_r, W1_r, H_r, ws1))
        calls.append((p2, None, W2, last_out, H_r, W2_r, Y_r, ws2))
        h2d = sum(t.numel() * t.element_size() for t in (X, W1, W2))
        if wl.name == "mlp_pair_sp":
            Y_h = torch.empty(tuple(wl.sp_out[0].shape), dtype=wl.sp_out[0].dtype).pin_memory()
            final_copy = (Y_h, wl.sp_out[0])
            d2h = Y_h.numel() * Y_h.element_size()
        else:
            d2h = last_out.numel() * last_out.element_size()
    else:
        A, B = (pin(t) for t in wl.host_globals)
        for p, A_r, B_r, C_r, ws in specs:
            dt = C_r[0].dtype
            C_h = torch.empty(p.shape[0], p.shape[2], dtype=dt).pin_memory()
            calls.append((p, A, B, C_h, A_r, B_r, C_r, ws))
            eb = A.element_size()
            h2d += _distinct_bytes(p, s.TENSOR_A, eb) + _distinct_bytes(p, s.TENSOR_B, eb)
            d2h += _distinct_bytes(p, s.TENSOR_C, C_h.element_size())

    def one_step():
        for p, A_h, B_h, C_h, A_r, B_r, C_r, ws in calls:
            p.run_host(A_h, B_h, C_h, A_r, B_r, C_r, ws, stream=stream)
        if wl.name == "mlp_pair_sp":
            wl.sp_gather.layernorm_all_gather(specs[-1][3], wl.sp_gamma, wl.sp_beta, wl.sp_out, stream=stream)
        if final_copy is not None:
            final_copy[0].copy_(final_copy[1], non_blocking=True)

    for _ in range(2):
        one_step()
    torch.cuda.synchronize()
    s.shmm_sync_status(stream)
    # Several windows of `steps` back-to-back steps, each between two events:
    # the host link's rate moves between windows (one window at a third of
    # the usual rate was seen), so the caller reports the median window and
    # lists them all.
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    per_window = []
    for _ in range(windows):
        dist_ctx.barrier()
        t0.record(stream)
        for _ in range(steps):
            one_step()
        t1.record(stream)
        torch.cuda.synchronize()
        per_window.append(dist_ctx.max(t0.elapsed_time(t1)) / steps)
    s.shmm_sync_status(stream)
    return per_window, h2d, d2h


def time_collective(s, H, torch, op, G, mib, dtype, reps=20, tree=False, stream_rate=True):
    """Bandwidth of one standalone collective on {X:G} partial buffers of
    ``mib`` MiB per rank (the full logical array V per rank).

    Two timings.  ``ms_median``: one launch at a time, L2 flushed before each,
    the device kept busy while the host enqueues it, so the events bracket
    one collective's device time including its launch.  ``stream_ms``: the
    collective over rotating buffer sets (together more than twice the L2,
    so no launch finds its inputs in L2 from an earlier one), launched back to
    back from a captured CUDA graph; the time per launch is the rate a stream
    of collectives sustains, with each launch's start overlapping the
    previous one's end.  CUDA events on this GPU tick in steps of about 2 us,
    which a graph of 32 or more launches averages out."""
    eb = 4 if dtype == "f32" else 2
    numel = int(mib * (1 << 20)) // eb
    cols = 4096 if numel >= 4096 * 16 else 256
    rows = numel // cols
    mesh = [("X", G)]
    fl = s.FLAG_PARTIAL_OUT_DTYPE | (s.FLAG_TREE if tree else 0)
    tdt = H.TORCH_DTYPES[dtype]
    V = rows * cols * eb
    if op == "all_to_all":
        nbytes = 2 * V               # A[I, J_X] -> A[I_X, J]: each rank reads and writes its V/G once
    elif op in ("all_gather", "layernorm_all_gather"):
        nbytes = V + G * V           # read V (each shard once), write G copies of V
    else:
        nbytes = G * V + (V if op == "reduce_scatter" else G * V)

    def make_set():
        if op == "all_to_all":
            src = [torch.empty((rows, cols // G), dtype=tdt, device="cuda").uniform_(-1, 1) for _ in range(G)]
            dst = [torch.empty((rows // G, cols), dtype=tdt, device="cuda") for _ in range(G)]
            return lambda st=None: s.shmm_reshard(mesh, ((), ("X",)), (("X",), ()), rows, cols, dtype, src, dst,
                                                  stream=st)
        if op in ("all_gather", "layernorm_all_gather"):
            p = s.Plan(mesh, (("X",), ()), ((), ()), ((), ()), rows, 8, cols, dtype, dtype)
            src = [torch.empty((rows // G, cols), dtype=tdt, device="cuda").uniform_(-1, 1) for _ in range(G)]
            dst = H.alloc(p, s.TENSOR_C)
            if op == "all_gather":
                return lambda st=None: p.all_gather(s.TENSOR_C, src, dst, stream=st)
            # sequence parallelism's LayerNorm of each token row fused with the
            # all-gather (gamma, beta: cols fp32 each, read once per thread)
            gamma = torch.ones(cols, dtype=torch.float32, device="cuda")
            beta = torch.zeros(cols, dtype=torch.float32, device="cuda")
            return lambda st=None: p.layernorm_all_gather(src, gamma, beta, dst, stream=st)
        sC = (("X",), ()) if op == "reduce_scatter" else ((), ())
        p = s.Plan(mesh, ((), ("X",)), (("X",), ()), sC, rows, G, cols, dtype, dtype, fl)
        src = [torch.empty((rows, cols), dtype=tdt, device="cuda").uniform_(-1, 1) for _ in range(G)]
        dst = H.alloc(p, s.TENSOR_C)
        if op == "reduce_scatter":
            return lambda st=None: p.reduce_scatter(src, dst, stream=st)
        return lambda st=None: p.all_reduce(src, dst, stream=st)

    run = make_set()
    # L2 flush by READING a buffer twice the L2 size: clean lines, so no
    # write-back of the flush itself lands inside the timed kernel
    flush = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        flush.sum()
        # keep the device busy while the host enqueues the start event and the
        # collective (argument checks and marshalling take tens of
        # microseconds), so the events bracket the device's work alone
        torch.cuda._sleep(SLEEP_CYCLES)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    t = statistics.median(times)
    busbw_factor = {"all_reduce": 2 * (G - 1) / G, "all_to_all": (G - 1) / G / 4}.get(op, (G - 1) / G)
    # off-rank bytes each rank sends, counted once at the sender ("Sharded
    # matmuls and collectives on a torus", payload accounting): RS and AG
    # (G-1)/G of V, AR both, all-to-all (G-1)/G of the rank's V/G
    payload = {"all_reduce": 2 * (G - 1) * V // G, "all_to_all": (G - 1) * V // (G * G)}.get(op, (G - 1) * V // G)
    out = {"op": op, "ranks": G, "MiB_per_rank": mib, "dtype": dtype, "order": "tree" if tree else "sequential",
           "ms_median": t, "ms_mean": statistics.mean(times), "ms_best": min(times),
           "GB_s": nbytes / (t * 1e-3) / 1e9,
           "l2_resident": G * V < 2 * L2_BYTES if op != "all_to_all" else V < 2 * L2_BYTES,
           "bytes": nbytes, "busbw_GB_s": (V / (t * 1e-3) / 1e9) * busbw_factor,
           "payload_bytes_per_rank": payload}
    if stream_rate:
        del run
        touched = nbytes  # bytes one launch reads and writes
        nsets = max(1, min(128, -(-4 * L2_BYTES // touched)))
        sets = [make_set() for _ in range(nsets)]
        launches = max(32, nsets)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for f in sets:
                f(side.cuda_stream)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream().cuda_stream
            for i in range(launches):
                sets[i % nsets](cs)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        st = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            b.synchronize()
            st.append(a.elapsed_time(b) / launches)
        ts = statistics.median(st)
        out.update({"stream_ms": ts, "stream_GB_s": nbytes / (ts * 1e-3) / 1e9, "stream_sets": nsets})
        del g, sets
    return out


# --------------------------------------------------------------- oracle

def _spread(n, k):
    """k row indices spread evenly over [0, n) (all rows when k >= n)."""
    if k >= n:
        return list(range(n))
    return sorted({int(i * n / k) for i in range(k)})


def _oracle_matmul(mesh, sA, sB, sC, A, B, out_dtype, rows, nthreads, gelu=False):
    """The oracle on sampled output rows; returns (per-rank result, FLOPs the
    sample took: each rank's local product over its sampled rows)."""
    import numpy as np
    import oracle
    _, res = oracle.sharded_matmul(mesh, sA, sB, sC, A, B, out_dtype=out_dtype, gelu=gelu, rows=rows,
                                   nthreads=nthreads)
    plan = oracle.plan_matmul(mesh, sA, sB, sC)
    I, J = A.shape
    K = B.shape[1]
    row_set = None if rows is None else np.asarray(sorted(set(rows)), np.int64)
    fl = 0
    for r in range(oracle.mesh_size(mesh)):
        (ai0, _), (ain, ajn) = oracle.shard_box(mesh, plan.local_A, (I, J), r)
        (_, _), (_, bkn) = oracle.shard_box(mesh, plan.local_B, (J, K), r)
        nr = ain if row_set is None else int(((row_set >= ai0) & (row_set < ai0 + ain)).sum())
        fl += 2 * nr * ajn * bkn
    return res, fl


def oracle_sample_step(cfg_name, rows_per_rank, nthreads, host_globals):
    """One bounded sample of the workload computed by the CPU oracle: about
    ``rows_per_rank`` output rows of every rank's block (local products,
    rank-order sum, rounding, ownership); the integer split-K case whole.
    Returns the sample's FLOPs."""
    import numpy as np
    import oracle
    c = WORKLOADS[cfg_name]
    if cfg_name in ("down_projection", "down_projection_quarter"):
        A, B = host_globals
        xs = dict(c["mesh"])["X"]
        blk = c["I"] // xs
        rows = sorted({x * blk + int(i * blk / rows_per_rank) for x in range(xs) for i in range(rows_per_rank)})
        return _oracle_matmul(c["mesh"], c["sA"], c["sB"], c["sC"], A, B, "bf16", rows, nthreads)[1]
    if cfg_name == "split_k_integer":
        A, B = host_globals
        return _oracle_matmul(c["mesh"], ((), ("Y",)), (("Y",), ()), (("Y",), ()), A, B, "f32", None, nthreads)[1]
    if cfg_name == "four_case":
        A, B = host_globals
        rows = _spread(c["I"], 4 * rows_per_rank)
        return sum(_oracle_matmul(c["mesh"], sA, sB, sC, A, B, "bf16", rows, nthreads)[1]
                   for sA, sB, sC in FOUR_CASES)
    if cfg_name in ("mlp_pair", "mlp_pair_sp"):
        # sampled tokens through both matmuls: H rows for those tokens, then
        # the second matmul (and for the sequence-parallel block its
        # reduce-scatter and LayerNorm) on them
        X, W1, W2 = host_globals
        mesh, T, D, F = c["mesh"], c["T"], c["D"], c["F"]
        n = oracle.mesh_size(mesh)
        t = _spread(T, max(n, (rows_per_rank * n) // n * n))
        t = t[:len(t) // n * n]
        res1, fl1 = _oracle_matmul(mesh, ((), ()), ((), ("X",)), ((), ("X",)), X, W1, "bf16", t, nthreads,
                                   gelu=True)
        H = np.zeros((len(t), F), np.float32)
        for r, (grows, k0, arr) in res1.items():
            H[:, k0:k0 + arr.shape[1]] = arr
        sC = (("X",), ()) if cfg_name == "mlp_pair_sp" else ((), ())
        res2, fl2 = _oracle_matmul(mesh, ((), ("X",)), (("X",), ()), sC, H, W2, "bf16", None, nthreads)
        if cfg_name == "mlp_pair_sp":
            for r, (off, y) in res2.items():
                oracle.layernorm(y, np.ones(D), np.zeros(D), 1e-5, out_dtype="bf16")
        return fl1 + fl2
    raise ValueError("no oracle sample for %s" % cfg_name)


def sample_text(cfg_name, rows, sample_flops, step_flops):
    if cfg_name == "split_k_integer":
        return "the whole step (%.3g MFLOP)" % (step_flops / 1e6)
    return ("about %d output rows of each rank's block (%.3g GFLOP of the step's %.4g GFLOP)"
            % (rows, sample_flops / 1e9, step_flops / 1e9))


def reference_host_globals(cfg_name):
    """The workload's global inputs as fp32 numpy arrays (the GPU arm's seeds)."""
    import shmm_inputs
    c = WORKLOADS[cfg_name]
    if cfg_name in ("mlp_pair", "mlp_pair_sp"):
        g = shmm_inputs.mlp_pair(c["T"], c["D"], c["F"], seed=0)
    elif cfg_name == "split_k_integer":
        g = shmm_inputs.split_k_integer(c["I"], c["J"], c["K"], seed=0)
    else:
        g = shmm_inputs.scaled_normal_pair(c["I"], c["J"], c["K"], "bf16", seed=0)
    return tuple(t.float().numpy() for t in g)


def full_step_flops(cfg_name):
    """FLOPs of one whole step of the workload, as the GPU arm counts them."""
    import oracle
    c = WORKLOADS[cfg_name]
    if cfg_name in ("mlp_pair", "mlp_pair_sp"):
        return 4.0 * c["T"] * c["D"] * c["F"]
    if cfg_name == "four_case":
        return float(oracle.mesh_size(c["mesh"]) *
                     sum(oracle.local_flops(c["mesh"], sA, sB, c["I"], c["J"], c["K"]) for sA, sB, _ in FOUR_CASES))
    return 2.0 * c["I"] * c["J"] * c["K"]


def oracle_reduce_scatter_gbs(nthreads, G=8, mib=16):
    """The oracle's reduce-scatter (ascending-rank fp32 sum, owner blocks) on
    G fp32 partial buffers of ``mib`` MiB, in GB/s by the GPU arm's byte
    count (G reads of V plus V written)."""
    import numpy as np
    import oracle
    n = mib * (1 << 20) // 4
    rng = np.random.default_rng(0)
    parts = [rng.uniform(-1, 1, (n // 4096, 4096)).astype(np.float32) for _ in range(G)]
    t0 = time.time()
    oracle.collective_reduce(parts, "reduce_scatter", "f32")
    dt = time.time() - t0
    return {"value": (G + 1) * n * 4 / dt / 1e9, "unit": "GB/s",
            "sample": "%d fp32 partials of %d MiB, reduce-scatter over rows" % (G, mib)}


def host_globals_f32(wl):
    return tuple(t.float().numpy() for t in wl.host_globals)


def cpu_baseline(cfg_name, host_globals, target_s=12.0):
    nthreads = len(os.sched_getaffinity(0))
    t0 = time.time()
    oracle_sample_step(cfg_name, 8, nthreads, host_globals)
    dt = time.time() - t0
    rows = max(8, min(1024, int(8 * target_s / max(dt, 1e-3))))
    t0 = time.time()
    fl = oracle_sample_step(cfg_name, rows, nthreads, host_globals)
    dt = time.time() - t0
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
            "sample": "%s, %.1f s" % (sample_text(cfg_name, rows, fl, full_step_flops(cfg_name)), dt),
            "reduce_scatter": oracle_reduce_scatter_gbs(nthreads)}


# ---------------------------------------------------------- distributed

class DistCtx:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            default = "nccl" if torch.cuda.is_available() else "gloo"
            backend = os.environ.get("SHMM_BENCH_BACKEND", default)
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, v):
        if self.pg is None:
            return v
        import torch
        dev = "cuda" if torch.cuda.is_available() and self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------ arms

def run_reference(args, dist_ctx):
    """The oracle on the host cores as the reference arm."""
    if dist_ctx.rank != 0:
        return None
    name = args.workload
    c = WORKLOADS[name]
    hg = reference_host_globals(name)
    nthreads = len(os.sched_getaffinity(0))
    budget = args.reference_budget_s / max(1, args.steps + args.warmup)
    t0 = time.time()
    oracle_sample_step(name, 1, nthreads, hg)
    one = time.time() - t0
    rows = max(1, min(256, int(budget / max(one, 1e-3))))
    for _ in range(args.warmup):
        oracle_sample_step(name, rows, nthreads, hg)
    t0 = time.time()
    fl = 0
    for _ in range(args.steps):
        fl += oracle_sample_step(name, rows, nthreads, hg)
    dt = time.time() - t0
    value = fl / dt / 1e12
    sample = sample_text(name, rows, fl / args.steps, full_step_flops(name)) + " per step"
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64-accumulate",
            "data": "synthetic", "config": {"workload": c["text"], "sample": sample},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
                             "sample": sample},
            "reduce_scatter": oracle_reduce_scatter_gbs(nthreads),
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_shmm(args, dist_ctx):
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: the shmm arm needs a CUDA device")
    torch.cuda.set_device(dist_ctx.local)
    from partial_sum_reduction_gb300 import build
    if dist_ctx.local == 0:
        build.build()
    dist_ctx.barrier()
    import partial_sum_reduction_gb300 as s
    from partial_sum_reduction_gb300 import helpers as H
    peaks, peak_kind = load_peaks()
    wl = Workload(args.workload, "cuda", rank_order=args.rank_order, sm_split=not args.no_sm_split,
                  batch=not args.no_batch)
    total_ms, per_step, launches, clocks = time_device(wl, args.steps, args.warmup, dist_ctx, graph=args.graph)
    ms = total_ms / args.steps
    N = dist_ctx.world
    value = wl.flops * N / (total_ms / args.steps * 1e-3) / 1e12
    # roofline of the dominant kernel: in the default workload one step is
    # one fused GEMM launch, so the per-step event time (the second loop,
    # an event pair around each step) is its duration
    launch_ms = statistics.mean(per_step)
    achieved = wl.flops / (launch_ms * 1e-3) / 1e12
    # The measured burst rate is the denominator for a kernel timed alone; a
    # kernel timed in a long back-to-back loop that ran under the power cap
    # (sw_power_cap during the timed region) is in the regime of the
    # measured sustained rate.  Both fractions are reported.
    power_capped = "sw_power_cap" in (clocks or {}).get("reasons", [])
    peak = peaks["bf16_tflops_sustained"] if power_capped else peaks["bf16_tflops"]
    e2e_steps = max(2, min(4, args.steps // 25))
    e2e_windows, h2d, d2h = time_e2e(wl, e2e_steps, dist_ctx)
    e2e_ms = statistics.median(e2e_windows)
    e2e_value = wl.flops * N / (e2e_ms * 1e-3) / 1e12
    rs = time_collective(s, H, torch, "reduce_scatter", 8, 256, "f32", stream_rate=False)
    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": N, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "ms_median_step": statistics.median(per_step),
        "ms_best_step": min(per_step), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload]["text"], "name": args.workload,
                   "launch": "CUDA graph replay" if args.graph else "direct shmm_run calls",
                   "four_case_launch": (None if args.workload != "four_case" else
                                        "shmm_run_batch: the four GEMMs in one launch" if wl.batch else
                                        "four streams, SMs split %s" % wl.sm_split if wl.sm_split else
                                        "four streams, whole-GPU launches"),
                   "fused_reduction": ("each rank's fp32 partial added in ascending rank order"
                                       if args.rank_order else
                                       "the group's products accumulated in one fp32 accumulator"),
                   "l2": "inputs larger than L2 (%.2f GB of per-rank operands per step)" % (wl.input_bytes() / 1e9),
                   "flop_per_step": wl.flops, "replicas": N},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "launch_ms": launch_ms,
                     "launch_timing": ("mean over a second loop of the same steps, each between its own "
                                       "pair of CUDA events on the launching stream"),
                     "traffic": kernel_traffic(args.workload),
                     "traffic_unit": "DRAM bytes per launch (ncu)",
                     "traffic_note": (NCU_TRAFFIC.get(args.workload, {}).get("note")
                                      if kernel_traffic(args.workload) else None),
                     "algorithmic_bytes": wl.input_bytes() + sum(t.numel() * t.element_size()
                                                                 for t in wl.output_tensors()),
                     "peak_kind": ("%s bf16 sustained (cuBLAS 8192^3 back to back): the timed loop ran under "
                                   "the power cap" % peak_kind if power_capped
                                   else "%s bf16 burst (cuBLAS 8192^3)" % peak_kind),
                     "frac_of_burst": achieved / peaks["bf16_tflops"],
                     "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                     "peak_nominal": NOMINAL_PEAKS["bf16_tflops"],
                     "frac_of_nominal": achieved / NOMINAL_PEAKS["bf16_tflops"],
                     "kernel": ("gemm_tc2_kernel (CTA pairs, 256x256 or 256x512 tiles as the launcher "
                                "picks) with fused reduction epilogue"
                                if os.environ.get("SHMM_TC_PAIR", "1") != "0"
                                else "gemm_tc_kernel<256> with fused reduction epilogue")},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "host_link_GB_s": (h2d + d2h) / (e2e_ms * 1e-3) / 1e9,
                "timing": "median of %d windows of %d steps (ms per step in ms_windows)" % (len(e2e_windows),
                                                                                           e2e_steps),
                "ms_windows": e2e_windows, "ms_mean": statistics.mean(e2e_windows),
                "note": ("shmm_run_host from pinned global host arrays: each distinct shard uploaded once, "
                         "replicas copied on the device, uploads/GEMMs/downloads pipelined by reduction "
                         "group; the global result written back to pinned host memory")},
        "gpu_launches": launches,
        "clocks": clocks,
        "reduce_scatter": {"value": rs["GB_s"], "unit": "GB/s", "frac": rs["GB_s"] / peaks["hbm_gbs"],
                           "peak": peaks["hbm_gbs"], "peak_kind": "%s HBM copy" % peak_kind,
                           "config": "fp32 partials, 8 ranks x 256 MiB, sequential rank order, L2 flushed",
                           "ms": rs["ms_median"], "ms_best": rs["ms_best"], "busbw_GB_s": rs["busbw_GB_s"],
                           "payload_bytes_per_rank": rs["payload_bytes_per_rank"],
                           "peak_nominal": NOMINAL_PEAKS["hbm_gbs"],
                           "frac_of_nominal": rs["GB_s"] / NOMINAL_PEAKS["hbm_gbs"]},
    }
    if dist_ctx.rank == 0 and N == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.workload, host_globals_f32(wl))
    return out


GEMM_SHAPES = [(8192, 8192, 2048), (8192, 8192, 8192), (8192, 8192, 16384), (16384, 16384, 2048),
               (2048, 8192, 14336), (8192, 4096, 16384)]


def run_gemm_sweep(args):
    """The local GEMM alone (one rank, no sharding) beside cuBLAS through
    torch.matmul on the same bf16 operands: CUDA events around batches of 10
    back-to-back launches, warm-up, median of 5 batches.  One JSON line per
    shape."""
    import torch
    from partial_sum_reduction_gb300 import build
    build.build()
    import partial_sum_reduction_gb300 as s
    peaks, kind = load_peaks()

    def med(fn, reps=5, batch=10):
        # batches of back-to-back launches between two events, so the host's
        # per-call cost overlaps the device work as in a real step loop
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts = []
        for _ in range(reps):
            a.record()
            for _ in range(batch):
                fn()
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b) / batch)
        return statistics.median(ts)

    for M, N, K in GEMM_SHAPES:
        A = torch.randn(M, K, device="cuda").to(torch.bfloat16)
        B = torch.randn(K, N, device="cuda").to(torch.bfloat16)
        C = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
        p = s.Plan([("X", 1)], ((), ()), ((), ()), ((), ()), M, K, N, "bf16", "bf16")
        f = 2.0 * M * N * K
        t_s = med(lambda: p.run([A], [B], [C]))
        t_c = med(lambda: torch.matmul(A, B, out=C))
        print(json.dumps({"gemm": [M, N, K], "shmm_tflops": f / t_s / 1e9, "cublas_tflops": f / t_c / 1e9,
                          "shmm_over_cublas": t_c / t_s, "frac_of_burst": f / t_s / 1e9 / peaks["bf16_tflops"],
                          "peak_kind": kind}), flush=True)
        del A, B, C


def run_sweep(args):
    import torch
    from partial_sum_reduction_gb300 import build
    build.build()
    import partial_sum_reduction_gb300 as s
    from partial_sum_reduction_gb300 import helpers as H
    peaks, kind = load_peaks()
    sizes = [float(x) if "." in x else int(x) for x in args.sizes.split(",")]
    ranks = [int(x) for x in args.ranks.split(",")]
    orders = {"sequential": (False,), "tree": (True,), "both": (False, True)}[args.orders]
    for op in args.ops.split(","):
        for dtype in args.dtypes.split(","):
            for G in ranks:
                for mib in sizes:
                    if G * mib * (2 if op == "all_reduce" else 1) > 40 * 1024:
                        continue
                    for tree in (orders if op in ("reduce_scatter", "all_reduce") else (False,)):
                        r = time_collective(s, H, torch, op, G, mib, dtype, reps=args.reps, tree=tree,
                                            stream_rate=not args.no_stream_rate)
                        r["frac_hbm"] = r["GB_s"] / peaks["hbm_gbs"]
                        if "stream_GB_s" in r:
                            r["stream_frac_hbm"] = r["stream_GB_s"] / peaks["hbm_gbs"]
                        r["peak_kind"] = kind
                        print(json.dumps(r), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="shmm", choices=["shmm", "reference"])
    ap.add_argument("--workload", default="down_projection", choices=sorted(WORKLOADS))
    ap.add_argument("--sweep", default=None, choices=[None, "collectives", "gemm"])
    ap.add_argument("--sizes", default="1,16,256,1024",
                    help="--sweep: MiB per rank (fractions allowed: 0.015625 is 16 KiB, the launch floor)")
    ap.add_argument("--ranks", default="2,4,8,16", help="--sweep collectives: group sizes")
    ap.add_argument("--ops", default="reduce_scatter,all_reduce,all_gather,all_to_all,layernorm_all_gather",
                    help="--sweep collectives: which collectives")
    ap.add_argument("--dtypes", default="f32,bf16", help="--sweep collectives: buffer types")
    ap.add_argument("--orders", default="both", choices=["sequential", "tree", "both"],
                    help="--sweep collectives: summation orders of RS and AR")
    ap.add_argument("--reps", type=int, default=20, help="--sweep collectives: single-launch repetitions")
    ap.add_argument("--no-stream-rate", action="store_true",
                    help="--sweep collectives: skip the back-to-back (graph-replayed) rate")
    ap.add_argument("--no-batch", action="store_true",
                    help="four_case: four shmm_run calls on four streams instead of one shmm_run_batch")
    ap.add_argument("--no-sm-split", action="store_true",
                    help="four_case: every case's GEMM may take all SMs (no split of the GPU among the cases)")
    ap.add_argument("--rank-order", action="store_true",
                    help="fused reductions add each rank's fp32 partial in ascending rank order "
                         "(SHMM_FLAG_RANK_ORDER) instead of accumulating the group in one accumulator")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="replay one captured CUDA graph per step (small workloads are host-bound)")
    ap.add_argument("--reference-budget-s", type=float, default=150.0,
                    help="--impl reference: seconds of oracle work for the whole run")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.sweep == "gemm":
        run_gemm_sweep(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    dist_ctx = DistCtx()
    try:
        if args.impl == "reference":
            out = run_reference(args, dist_ctx)
        else:
            out = run_shmm(args, dist_ctx)
        if dist_ctx.rank == 0 and out is not None:
            print(json.dumps(out), flush=True)
    finally:
        dist_ctx.close()


if __name__ == "__main__":
    main()
