"""The C-ABI library without a GPU: it builds, loads, exports every symbol
include/shmm.h declares, and its host planner agrees with the oracle's
independent box logic on every mesh/sharding combination tried.  Argument
checks and the injected-failure hook are exercised before any device call."""
import ctypes
import itertools
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def shmm():
    from partial_sum_reduction_gb300 import build
    build.build()
    import partial_sum_reduction_gb300 as s
    return s


def declared_functions():
    src = open(os.path.join(ROOT, "include", "shmm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(shmm_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(shmm):
    names = declared_functions()
    assert len(names) >= 15
    L = ctypes.CDLL(shmm.shmm.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(shmm.shmm.EXPORTS)
    assert shmm.shmm_version() == 100
    assert shmm.lib().shmm_status_string(0) == b"SHMM_OK"


def test_binding_constants_match_header(shmm):
    """Every SHMM_FLAG_*, SHMM_TENSOR_* and dtype value the header defines has
    the same value in the binding."""
    src = open(os.path.join(ROOT, "include", "shmm.h")).read()
    flags = dict(re.findall(r"#define SHMM_FLAG_([A-Z_]+) (0x[0-9a-fA-F]+)u", src))
    assert len(flags) >= 6
    for name, val in flags.items():
        assert getattr(shmm, "FLAG_" + name) == int(val, 16), name
    tensors = dict(re.findall(r"SHMM_TENSOR_([A-Z_]+) = (\d+)", src))
    assert len(tensors) == 7
    for name, val in tensors.items():
        assert getattr(shmm, "TENSOR_" + name) == int(val), name
    ws = re.search(r"#define SHMM_STATIC_WORKSPACE_BYTES \((\d+)u << (\d+)\)", src)
    assert shmm.shmm.STATIC_WORKSPACE_BYTES == int(ws.group(1)) << int(ws.group(2))
    assert (shmm.F32, shmm.BF16) == (0, 1)


def test_binding_status_codes_match_header(shmm):
    """Every status code the header defines has the binding's value and the
    library's name."""
    src = open(os.path.join(ROOT, "include", "shmm.h")).read()
    codes = dict(re.findall(r"SHMM_(OK|ERR_[A-Z_]+) = (\d+)", src))
    assert len(codes) == 13
    for name, val in codes.items():
        assert getattr(shmm.shmm, name) == int(val), name
        assert shmm.lib().shmm_status_string(int(val)).decode() == "SHMM_" + name


def test_bounds_checked_build_exports_every_declared_symbol(shmm):
    """The bounds-checked variant (same sources, SHMM_CHECKED) builds, exports
    the same C ABI and says which build it is; the ordinary one says not."""
    from partial_sum_reduction_gb300 import build
    L = ctypes.CDLL(build.build(checked=True))
    for n in declared_functions():
        assert hasattr(L, n), n
    assert L.shmm_bounds_checked() == 1
    assert ctypes.CDLL(build.LIB).shmm_bounds_checked() == 0


def test_every_environment_knob_is_documented():
    """Each variable the library reads with getenv is described in the
    header, so a user of the C ABI alone can find it."""
    import glob
    header = open(os.path.join(ROOT, "include", "shmm.h")).read()
    used = set()
    for f in glob.glob(os.path.join(ROOT, "partial_sum_reduction_gb300", "csrc", "*")):
        used |= set(re.findall(r'getenv\("(SHMM_[A-Z_]+)"\)', open(f).read()))
    assert used >= {"SHMM_TC_PAIR", "SHMM_TC_WIDE", "SHMM_INJECT_FAIL"}
    for name in used:
        assert name in header, name


def test_binding_fails_loudly_without_library(monkeypatch):
    import partial_sum_reduction_gb300.shmm as m
    monkeypatch.setattr(m, "_lib", None)
    monkeypatch.setattr(m, "LIB_PATH", "/nonexistent/libshmm.so")
    with pytest.raises(RuntimeError):
        m.lib()


MESHES = {
    "Y2": [("Y", 2)],
    "XY22": [("X", 2), ("Y", 2)],
    "XY42": [("X", 4), ("Y", 2)],
    "X8": [("X", 8)],
    "XYZ222": [("X", 2), ("Y", 2), ("Z", 2)],
}


def specs_for(mesh):
    names = [n for n, _ in mesh]
    dims = [()] + [(a,) for a in names] + [tuple(p) for p in itertools.permutations(names, 2)]
    return dims


def all_combos():
    rng = np.random.default_rng(0)
    out = []
    for mname, mesh in MESHES.items():
        dims = specs_for(mesh)
        for _ in range(60):
            sA = (dims[rng.integers(len(dims))], dims[rng.integers(len(dims))])
            sB = (dims[rng.integers(len(dims))], dims[rng.integers(len(dims))])
            sC = (dims[rng.integers(len(dims))], dims[rng.integers(len(dims))])
            out.append((mname, sA, sB, sC))
    # the workloads' own shardings
    out += [("Y2", ((), ("Y",)), (("Y",), ()), (("Y",), ())),
            ("XY22", (("X",), ()), ((), ("Y",)), (("X",), ("Y",))),
            ("XY22", ((), ("X",)), ((), ()), ((), ())),
            ("XY22", ((), ("Y",)), (("Y",), ()), (("Y",), ())),
            ("XY22", (("X",), ()), ((), ("X",)), (("X",), ())),
            ("X8", ((), ()), ((), ("X",)), ((), ("X",))),
            ("X8", ((), ("X",)), (("X",), ()), ((), ())),
            ("X8", ((), ("X",)), (("X",), ()), (("X",), ())),
            ("XY42", (("X",), ("Y",)), (("Y",), ()), (("X",), ()))]
    return out


@pytest.mark.parametrize("mname,sA,sB,sC", all_combos())
def test_planner_matches_oracle(shmm, mname, sA, sB, sC):
    mesh = MESHES[mname]
    I, J, K = 48, 96, 24
    try:
        oplan = oracle.plan_matmul(mesh, sA, sB, sC)
        for spec, shape in ((sA, (I, J)), (sB, (J, K)), (sC, (I, K)), (oplan.reduced_C, (I, K))):
            oracle.shard_box(mesh, spec, shape, 0)
        oerr = None
    except ValueError as e:
        oerr = e
    try:
        p = shmm.Plan(mesh, sA, sB, sC, I, J, K, "bf16", "bf16")
        perr = None
    except shmm.ShmmError as e:
        perr = e
    assert (oerr is None) == (perr is None), (oerr, perr)
    if oerr is not None:
        return
    info = p.info
    assert info.case_id == oplan.case
    assert shmm.shmm.COLLECTIVE_NAMES[info.collective] == oplan.collective
    assert info.scatter_dim == oplan.scatter_dim
    N = oracle.mesh_size(mesh)
    T = shmm
    for r in range(N):
        for tensor, spec, shape in ((T.TENSOR_A, sA, (I, J)), (T.TENSOR_B, sB, (J, K)),
                                    (T.TENSOR_C, sC, (I, K)), (T.TENSOR_P, oplan.natural_C, (I, K)),
                                    (T.TENSOR_A_LOCAL, oplan.local_A, (I, J)),
                                    (T.TENSOR_B_LOCAL, oplan.local_B, (J, K)),
                                    (T.TENSOR_C_REDUCED, oplan.reduced_C, (I, K))):
            assert p.rank_box(tensor, r) == oracle.shard_box(mesh, spec, shape, r), (tensor, r)
        if info.group_size > 1:
            assert p.group(r) == oracle.reduction_group(mesh, oplan, r)
    pay = oracle.payload_bytes(mesh, sA, sB, sC, I, J, K, "bf16", "bf16")
    assert info.payload_operand_ag == pay["operand_all_gather"]
    assert info.payload_reduce_scatter == pay["reduce_scatter"]
    assert info.payload_result_ag == pay["result_all_gather"]
    assert info.flops_per_rank == oracle.local_flops(mesh, sA, sB, I, J, K)


def test_worked_example_plan(shmm, golden):
    g = golden("p2_worked_example.txt")
    p = shmm.Plan("{Y:2}", "I,J_Y", "J_Y,K", "I_Y,K", 2, 2, 2, "f32", "f32")
    assert p.info.payload_reduce_scatter == g["reduce_scatter_payload_bytes_per_rank"]
    p = shmm.Plan("{Y:2}", "I,J_Y", "J_Y,K", "I,K", 2, 2, 2, "f32", "f32")
    assert p.info.payload_reduce_scatter + p.info.payload_result_ag == g["payload_bytes_per_rank"]
    assert (p.info.payload_reduce_scatter + p.info.payload_result_ag) * 2 == g["payload_bytes_total"]


def test_down_projection_plan(shmm, golden):
    g = golden("p4_down_projection.txt")
    p = shmm.Plan("{X:4,Y:2}", "P('X','Y')", "P('Y',None)", "P('X',None)", 8192, 28672, 8192,
                  "bf16", "bf16", shmm.FLAG_FUSED)
    assert list(p.rank_box(shmm.TENSOR_A, 0)[1]) == g["A_shard"]
    assert round(p.info.flops_per_rank / 1e9) == g["local_matmul_GFLOP"]
    assert p.info.case_id == 3 and p.info.group_size == 2 and p.info.tensor_core == 1
    assert p.info.fused == 1 and p.info.workspace_bytes == 0
    _, ext = p.rank_box(shmm.TENSOR_C, 0)
    assert round(ext[0] * ext[1] * 2 / 1e6, 1) == g["C_bytes_per_device_MB"]


def test_spec_string_forms(shmm):
    assert shmm.parse_spec("P(('X','Y'),None)") == (("X", "Y"), ())
    assert shmm.parse_spec("P('X', 'Y')") == (("X",), ("Y",))
    assert shmm.parse_spec("P()") == ((), ())
    assert shmm.parse_spec("P(None,'Y')") == ((), ("Y",))
    assert shmm.parse_spec("I_XY,J") == (("X", "Y"), ())
    assert shmm.parse_mesh("{X:4,Y:2}") == [("X", 4), ("Y", 2)]


@pytest.mark.parametrize("bad,code", [
    (("{X:2}", "I_X,J_X", "J,K", "I,K", 4, 4, 4), "ERR_INVALID_SPEC"),
    (("{X:2}", "I_X,J", "J,K_X", "I_X,K_X", 4, 4, 4), "ERR_ILLEGAL_OUTPUT"),
    (("{X:2}", "I_Z,J", "J,K", "I,K", 4, 4, 4), "ERR_INVALID_SPEC"),
    (("{X:2}", "I_X,J", "J,K", "I,K", 3, 4, 4), "ERR_SHAPE"),
    (("{X:2}", "I,J", "J,K", "I,K", -1, 4, 4), "ERR_SHAPE"),
    (("{X:2}", "I,J_X", "J_X,K", "I_X,K_X", 4, 4, 4), "ERR_ILLEGAL_OUTPUT"),
    (("{X:2,Y:2}", "I,J_XY", "J_XY,K", "I_X,K_Y", 4, 4, 4), "ERR_INVALID_SPEC"),
    (("{X:2,Y:2}", "I,J_X", "J_X,K", "I_Y,K", 4, 4, 4), "ERR_INVALID_SPEC"),
    (("{X:300}", "I,J", "J,K", "I,K", 4, 4, 4), "ERR_SHAPE"),
])
def test_plan_rejections(shmm, bad, code):
    with pytest.raises(shmm.ShmmError) as e:
        shmm.Plan(*bad)
    assert e.value.status == getattr(shmm.shmm, code)


def test_argument_checks_before_any_device_call(shmm, monkeypatch):
    """NULL, misaligned and undersized arguments, and the injected failure,
    return their status without touching the GPU (this runs on CPU)."""
    p = shmm.Plan("{Y:2}", "I,J_Y", "J_Y,K", "I_Y,K", 64, 64, 64, "bf16", "bf16")
    L = shmm.lib()
    PP = ctypes.c_void_p * 2
    good = PP(0x10000, 0x20000)
    bad_align = PP(0x10000, 0x20008)
    nulls = PP(0, 0)
    assert L.shmm_local_matmul(p.handle, None, good, good, None) == shmm.shmm.ERR_NULL
    assert L.shmm_local_matmul(p.handle, nulls, good, good, None) == shmm.shmm.ERR_NULL
    assert L.shmm_local_matmul(p.handle, good, bad_align, good, None) == shmm.shmm.ERR_ALIGN
    assert b"16-byte" in L.shmm_last_error()
    assert L.shmm_reduce_scatter(p.handle, good, bad_align, None) == shmm.shmm.ERR_ALIGN
    assert L.shmm_all_gather(p.handle, shmm.TENSOR_A, good, good, None) == shmm.shmm.ERR_UNSUPPORTED
    assert L.shmm_all_gather(p.handle, 9, good, good, None) == shmm.shmm.ERR_UNSUPPORTED
    p1 = shmm.Plan("{Y:2}", "I_Y,J", "J,K", "I_Y,K", 64, 64, 64, "bf16", "bf16")
    assert L.shmm_all_reduce(p1.handle, good, good, None) == shmm.shmm.ERR_UNSUPPORTED
    pr = shmm.Plan("{Y:2}", "I,J_Y", "J_Y,K", "I_Y,K", 64, 64, 64, "bf16", "bf16")
    assert pr.workspace_size() == 2 * 64 * 64 * 4
    assert L.shmm_run(pr.handle, good, good, good, None, 0, None) == shmm.shmm.ERR_NOMEM
    assert L.shmm_run(pr.handle, good, good, good, ctypes.c_void_p(0x100080), 1 << 20, None) == \
        shmm.shmm.ERR_ALIGN
    assert L.shmm_run(None, good, good, good, None, 0, None) == shmm.shmm.ERR_NULL
    # shmm_run_host checks the same arguments before any copy is enqueued
    h = ctypes.c_void_p(0x30000)
    assert L.shmm_run_host(None, h, h, h, good, good, good, None, 0, None) == shmm.shmm.ERR_NULL
    assert L.shmm_run_host(pr.handle, h, h, h, nulls, good, good, None, 0, None) == shmm.shmm.ERR_NULL
    assert L.shmm_run_host(pr.handle, h, h, h, good, bad_align, good, None, 0, None) == shmm.shmm.ERR_ALIGN
    assert L.shmm_run_host(pr.handle, h, h, h, good, good, good, None, 0, None) == shmm.shmm.ERR_NOMEM
    import torch
    for bad in (np.zeros((64, 64)), torch.zeros(64, 32), torch.zeros(64, 128)[:, :64]):
        with pytest.raises(ValueError):
            pr.run_host(bad, None, None, [0x10000] * 2, [0x10000] * 2, [0x10000] * 2)
    monkeypatch.setenv("SHMM_INJECT_FAIL", "shmm_run,shmm_all_reduce,shmm_run_host")
    assert L.shmm_run_host(pr.handle, h, h, h, good, good, good, None, 0, None) == shmm.shmm.ERR_INJECTED
    assert L.shmm_run(pr.handle, good, good, good, None, 0, None) == shmm.shmm.ERR_INJECTED
    assert L.shmm_all_reduce(pr.handle, good, good, None) == shmm.shmm.ERR_INJECTED
    assert b"injected" in L.shmm_last_error()
    with pytest.raises(shmm.ShmmError) as e:
        pr.run([0x10000, 0x20000], [0x10000, 0x20000], [0x10000, 0x20000], stream=0)
    assert e.value.status == shmm.shmm.ERR_INJECTED


def test_workspace_accounting(shmm):
    # case 2: A gathered per rank; case 3 unfused: fp32 partials; fused: none
    p = shmm.Plan("{X:2,Y:2}", "I,J_X", "J,K", "I,K", 256, 256, 128, "bf16", "bf16")
    assert p.workspace_size() == 4 * 256 * 256 * 2
    p = shmm.Plan("{X:2,Y:2}", "I,J_Y", "J_Y,K", "I_Y,K", 256, 256, 128, "bf16", "bf16")
    assert p.workspace_size() == 4 * 256 * 128 * 4
    p = shmm.Plan("{X:2,Y:2}", "I,J_Y", "J_Y,K", "I_Y,K", 256, 256, 128, "bf16", "bf16", shmm.FLAG_FUSED)
    assert p.workspace_size() == 0 and p.info.fused == 1
    # up to 16 ranks per group fuse on the tensor cores; more reduce unfused
    p = shmm.Plan("{X:16}", "I,J_X", "J_X,K", "I,K", 256, 256, 128, "bf16", "bf16", shmm.FLAG_FUSED)
    assert p.info.fused == 1 and p.workspace_size() == 0
    p = shmm.Plan("{X:32}", "I,J_X", "J_X,K", "I,K", 256, 256, 128, "bf16", "bf16", shmm.FLAG_FUSED)
    assert p.info.fused == 0 and p.workspace_size() == 32 * 256 * 128 * 4


def test_in_place_gather_decision(shmm):
    """SHMM_FLAG_FUSED reads case 2/4 operands from their owners' shards when
    every TMA box lies inside one shard; otherwise the all-gather stays."""
    F = shmm.FLAG_FUSED
    p = shmm.Plan("{X:2,Y:2}", "I,J_X", "J,K", "I,K", 256, 256, 128, "bf16", "bf16", F)
    assert p.info.fused_gather == 1 and p.workspace_size() == 0
    p = shmm.Plan("{X:2,Y:2}", "I_X,J", "J,K_X", "I_X,K", 256, 256, 256, "bf16", "bf16", F)
    assert p.info.case_id == 4 and p.info.fused_gather == 1 and p.workspace_size() == 0
    # shard width 96 (not a multiple of 64): gather into the workspace
    p = shmm.Plan("{X:2,Y:2}", "I,J_X", "J,K", "I,K", 256, 192, 128, "bf16", "bf16", F)
    assert p.info.fused_gather == 0 and p.workspace_size() == 4 * 256 * 192 * 2
    # without the flag, or off the tensor cores, nothing fuses
    p = shmm.Plan("{X:2,Y:2}", "I,J_X", "J,K", "I,K", 256, 256, 128, "bf16", "bf16")
    assert p.info.fused_gather == 0
    p = shmm.Plan("{X:2,Y:2}", "I,J_X", "J,K", "I,K", 256, 256, 128, "f32", "f32", F)
    assert p.info.fused_gather == 0
    # case 3 and case 4 at once: reduction and gather both fused
    p = shmm.Plan("{X:2,Y:2}", "I_X,J_Y", "J_Y,K_X", "I_X,K", 512, 256, 256, "bf16", "bf16", F)
    assert p.info.case_id == 3 and p.info.fused == 1 and p.info.fused_gather == 1
    assert p.workspace_size() == 0


def test_operand_choice_reproduces_the_pages_thresholds(shmm, golden):
    """Strategy 1 (gather W) is compute-bound when B > C/W; at large B
    strategy 2 (reduce the [B,F] partials) wins exactly when D > 2C/W."""
    g = golden("p4_operand_choice.txt")
    for chip in ("v5p_book", "v5p_docs", "ironwood"):
        W = g[chip + "_W"]
        C = g[chip + "_intensity"] * W
        thr = g[chip + "_threshold"]
        assert thr == 2 * g[chip + "_intensity"]
        F, n, Bbig = 8192, 4, 10 ** 8
        assert shmm.shmm_choose_operand(Bbig, thr - 10, F, n, C, W).choice == 1
        assert shmm.shmm_choose_operand(Bbig, thr + 10, F, n, C, W).choice == 2
        ci = g[chip + "_intensity"]
        assert shmm.shmm_choose_operand(ci - 5, 4096, F, n, C, W).gather_compute_bound == 0
        assert shmm.shmm_choose_operand(ci + 5, 4096, F, n, C, W).gather_compute_bound == 1
    r = shmm.shmm_choose_operand(1024, 4096, 16384, 4, 1e15, 1e11)
    assert r.bytes_gather == g["strategy1_bytes_per_DF"] * 4096 * 16384
    assert r.bytes_reduce == g["strategy2_bytes_per_BF"] * 1024 * 16384
    with pytest.raises(shmm.ShmmError):
        shmm.shmm_choose_operand(0, 1, 1, 2, 1e15, 1e11)


def test_reshard_argument_checks(shmm, monkeypatch):
    import ctypes
    good = [0x10000, 0x20000]
    with pytest.raises(shmm.ShmmError) as e:
        shmm.shmm_reshard("{X:2}", "I,J_X", "I_X,J_X", 4, 4, "f32", good, good, stream=0)
    assert e.value.status == shmm.shmm.ERR_INVALID_SPEC
    with pytest.raises(shmm.ShmmError) as e:
        shmm.shmm_reshard("{X:2}", "I,J_X", "I_X,J", 3, 4, "f32", good, good, stream=0)
    assert e.value.status == shmm.shmm.ERR_SHAPE
    with pytest.raises(shmm.ShmmError) as e:
        shmm.shmm_reshard("{X:2}", "I,J_X", "I_X,J", 4, 4, "f32", [0x10000, 0], good, stream=0)
    assert e.value.status == shmm.shmm.ERR_NULL
    with pytest.raises(shmm.ShmmError) as e:
        shmm.shmm_reshard("{X:2}", "I,J_X", "I_X,J", 4, 4, "f32", good, [0x10000, 0x20004], stream=0)
    assert e.value.status == shmm.shmm.ERR_ALIGN
    monkeypatch.setenv("SHMM_INJECT_FAIL", "shmm_reshard")
    with pytest.raises(shmm.ShmmError) as e:
        shmm.shmm_reshard("{X:2}", "I,J_X", "I_X,J", 4, 4, "f32", good, good, stream=0)
    assert e.value.status == shmm.shmm.ERR_INJECTED


def test_sm_limit_argument_checks(shmm):
    p = shmm.Plan("{X:2,Y:2}", "I_X,J", "J,K_Y", "I_X,K_Y", 512, 256, 512, "bf16", "bf16")
    p.set_sm_limit(32)
    p.set_sm_limit(0)
    with pytest.raises(shmm.ShmmError) as e:
        p.set_sm_limit(-1)
    assert e.value.status == shmm.shmm.ERR_SHAPE
    assert shmm.lib().shmm_plan_set_sm_limit(None, 4) == shmm.shmm.ERR_NULL


def test_run_batch_argument_checks(shmm):
    """Every plan and pointer is checked before anything is enqueued; the
    message names the offending plan."""
    L = shmm.lib()
    import ctypes
    PP = ctypes.POINTER(ctypes.c_void_p)
    assert L.shmm_run_batch(0, None, None, None, None, None, None, None) == shmm.shmm.OK
    assert L.shmm_run_batch(-1, None, None, None, None, None, None, None) == shmm.shmm.ERR_SHAPE
    assert L.shmm_run_batch(1, None, None, None, None, None, None, None) == shmm.shmm.ERR_NULL
    p0 = shmm.Plan("{X:2,Y:2}", "I_X,J", "J,K_Y", "I_X,K_Y", 512, 256, 512, "bf16", "bf16")
    p1 = shmm.Plan("{X:2,Y:2}", "I,J_Y", "J_Y,K", "I_Y,K", 512, 256, 512, "bf16", "bf16", shmm.FLAG_FUSED)
    good = (ctypes.c_void_p * 4)(*([0x10000] * 4))
    bad = (ctypes.c_void_p * 4)(*([0x10008] * 4))   # not 16-byte aligned
    handles = (ctypes.c_void_p * 2)(p0.handle.value, p1.handle.value)
    g = ctypes.cast(good, PP)
    b = ctypes.cast(bad, PP)
    A = (PP * 2)(g, g)
    B = (PP * 2)(g, b)
    C = (PP * 2)(g, g)
    assert L.shmm_run_batch(2, handles, A, B, C, None, None, None) == shmm.shmm.ERR_ALIGN
    assert b"plan 1" in L.shmm_last_error()
    handles_null = (ctypes.c_void_p * 2)(p0.handle.value, None)
    assert L.shmm_run_batch(2, handles_null, A, A, C, None, None, None) == shmm.shmm.ERR_NULL
