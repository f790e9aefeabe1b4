"""shmm_run_host: global operands in host memory -> the ranks' device shards
-> the sharded matmul -> the global result in host memory.  Every device
buffer it fills and every host element it writes must be bit for bit what
uploading the shards and calling shmm_run gives."""
import numpy as np
import pytest
import torch

import shmm_inputs
from parity_util import F32P_TOL, compare, lib, oracle_run

pytestmark = pytest.mark.gpu

Y2 = [("Y", 2)]
XY22 = [("X", 2), ("Y", 2)]
XY42 = [("X", 4), ("Y", 2)]
X8 = [("X", 8)]

# (name, mesh, sA, sB, sC, I, J, K, flags, staged)
PLANS = [
    ("fused_AR_4_groups", XY42, (("X",), ("Y",)), (("Y",), ()), (("X",), ()), 1024, 1024, 384, "FUSED", True),
    ("fused_RS_rows", X8, ((), ("X",)), (("X",), ()), (("X",), ()), 512, 1024, 256, "FUSED", True),
    ("fused_RS_cols", [("X", 4)], ((), ("X",)), (("X",), ()), ((), ("X",)), 384, 512, 512, "FUSED", True),
    ("case1_no_reduction", XY22, (("X",), ()), ((), ("Y",)), (("X",), ("Y",)), 512, 384, 512, "0", True),
    ("replicated_A_gelu", X8, ((), ()), ((), ("X",)), ((), ("X",)), 256, 512, 1024, "GELU", True),
    ("case2_gather", XY22, ((), ("X",)), ((), ()), ((), ()), 384, 512, 264, "0", False),
    ("unfused_AR", Y2, ((), ("Y",)), (("Y",), ()), ((), ()), 256, 512, 320, "0", False),
    ("fused_then_replicate", XY22, ((), ("Y",)), (("Y",), ()), ((), ()), 256, 512, 320, "FUSED", True),
    # Host operands of >= 32 MB run in one stage per 16 MB; with fewer units
    # than that, each unit's stage splits into blocks of output rows.
    # One reduction group, 84 MB: five row blocks of 1024, the last 4 rows.
    ("row_blocks_fused_AR", Y2, ((), ("Y",)), (("Y",), ()), ((), ()), 4100, 8192, 1024, "FUSED", True),
    # A replicated over both ranks, 53 MB: two blocks per rank, and rank 1's
    # blocks are device copies of rank 0's
    ("row_blocks_replicated_A", [("X", 2)], ((), ()), ((), ("X",)), ((), ("X",)), 6000, 4096, 512, "0", True),
    # rank-order fold, reduce-scatter over columns, 57 MB: three row blocks
    ("row_blocks_RS_cols_rank_order", Y2, ((), ("Y",)), (("Y",), ()), ((), ("Y",)), 3000, 8192, 512,
     "FUSED|RANK_ORDER", True),
]


@pytest.fixture(scope="module")
def s():
    assert torch.cuda.is_available()
    return lib()


def _flags(s, names):
    fl = 0
    for f in names.split("|"):
        fl |= getattr(s, "FLAG_" + f) if f != "0" else 0
    return fl


def _stitch(plan, s, C_r, I, K, dtype):
    """The global C from the ranks' blocks (every element covered)."""
    out = torch.full((I, K), float("nan"), dtype=dtype)
    for r, c in enumerate(C_r):
        (o0, o1), (e0, e1) = plan.rank_box(s.TENSOR_C, r)
        out[o0:o0 + e0, o1:o1 + e1] = c.cpu()
    return out


@pytest.mark.parametrize("name,mesh,sA,sB,sC,I,J,K,flags,staged", PLANS, ids=[p[0] for p in PLANS])
@pytest.mark.parametrize("pinned", [True, False])
def test_run_host_equals_device_path(s, name, mesh, sA, sB, sC, I, J, K, flags, staged, pinned):
    from partial_sum_reduction_gb300 import helpers as H
    A, B = shmm_inputs.scaled_normal_pair(I, J, K, "bf16", seed=I + K)
    plan = s.Plan(mesh, sA, sB, sC, I, J, K, "bf16", "bf16", _flags(s, flags))
    # the device path
    A_d, B_d = H.shard(plan, s.TENSOR_A, A), H.shard(plan, s.TENSOR_B, B)
    C_d = H.alloc(plan, s.TENSOR_C, fill=float("nan"))
    ws = H.workspace(plan)
    plan.run(A_d, B_d, C_d, ws)
    # from host memory into fresh device buffers
    A_h, B_h = (A.pin_memory(), B.pin_memory()) if pinned else (A.clone(), B.clone())
    C_h = torch.full((I, K), float("nan"), dtype=torch.bfloat16)
    if pinned:
        C_h = C_h.pin_memory()
    A_r = H.alloc(plan, s.TENSOR_A, fill=float("nan"))
    B_r = H.alloc(plan, s.TENSOR_B, fill=float("nan"))
    C_r = H.alloc(plan, s.TENSOR_C, fill=float("nan"))
    plan.run_host(A_h, B_h, C_h, A_r, B_r, C_r, ws)
    s.shmm_sync_status()
    torch.cuda.synchronize()
    for x, y in zip(A_r + B_r, A_d + B_d):
        assert torch.equal(x, y)
    for x, y in zip(C_r, C_d):
        assert torch.equal(x, y)
    assert not torch.isnan(C_h).any(), "an element of the host result was not written"
    assert torch.equal(C_h, _stitch(plan, s, C_d, I, K, torch.bfloat16))


def test_run_host_staged_matches_oracle(s):
    """The staged path (four reduction groups, four stages) against the
    oracle, fp32 result."""
    mesh, sA, sB, sC = XY42, (("X",), ("Y",)), (("Y",), ()), (("X",), ())
    I, J, K = 1024, 1024, 384
    A, B = shmm_inputs.scaled_normal_pair(I, J, K, "bf16", seed=21)
    from partial_sum_reduction_gb300 import helpers as H
    plan = s.Plan(mesh, sA, sB, sC, I, J, K, "bf16", "f32", s.FLAG_FUSED)
    C_h = torch.full((I, K), float("nan"), dtype=torch.float32).pin_memory()
    A_r, B_r = H.alloc(plan, s.TENSOR_A), H.alloc(plan, s.TENSOR_B)
    C_r = H.alloc(plan, s.TENSOR_C, fill=float("nan"))
    plan.run_host(A.pin_memory(), B.pin_memory(), C_h, A_r, B_r, C_r)
    s.shmm_sync_status()
    torch.cuda.synchronize()
    _, ores = oracle_run(mesh, sA, sB, sC, A, B, "f32")
    compare(plan, [c.cpu() for c in C_r], ores, exact=False, tol=F32P_TOL)
    for r in range(plan.nranks):
        (o0, o1), blk = ores[r]
        np.testing.assert_array_equal(C_h[o0:o0 + blk.shape[0], o1:o1 + blk.shape[1]].numpy(),
                                      C_r[r].cpu().numpy())


def test_run_host_null_operands_and_chained_calls(s):
    """A NULL host operand means the shards are already on the device (the
    MLP pair keeps its intermediate there); a NULL C_host leaves the result
    on the device.  Two calls on one stream: the second's uploads wait for
    the first's GEMMs."""
    from partial_sum_reduction_gb300 import helpers as H
    T, D, F = 256, 512, 1024
    X, W1, W2 = shmm_inputs.mlp_pair(T, D, F, seed=7)
    p1 = s.Plan(X8, ((), ()), ((), ("X",)), ((), ("X",)), T, D, F, "bf16", "bf16", s.FLAG_GELU)
    p2 = s.Plan(X8, ((), ("X",)), (("X",), ()), ((), ()), T, F, D, "bf16", "bf16", s.FLAG_FUSED)
    # device path
    H_d = H.alloc(p1, s.TENSOR_C)
    p1.run(H.shard(p1, s.TENSOR_A, X), H.shard(p1, s.TENSOR_B, W1), H_d)
    Y_d = H.alloc(p2, s.TENSOR_C)
    p2.run(H_d, H.shard(p2, s.TENSOR_B, W2), Y_d)
    # host path: X, W1 in; H stays on the device; W2 in, Y out
    X_r, W1_r, H_r = H.alloc(p1, s.TENSOR_A), H.alloc(p1, s.TENSOR_B), H.alloc(p1, s.TENSOR_C, fill=float("nan"))
    p1.run_host(X.pin_memory(), W1.pin_memory(), None, X_r, W1_r, H_r)
    W2_r, Y_r = H.alloc(p2, s.TENSOR_B), H.alloc(p2, s.TENSOR_C, fill=float("nan"))
    Y_h = torch.full((T, D), float("nan"), dtype=torch.bfloat16).pin_memory()
    p2.run_host(None, W2.pin_memory(), Y_h, H_r, W2_r, Y_r)
    s.shmm_sync_status()
    torch.cuda.synchronize()
    for x, y in zip(H_r, H_d):
        assert torch.equal(x, y)
    for x, y in zip(Y_r, Y_d):
        assert torch.equal(x, y)
    assert torch.equal(Y_h, Y_d[0].cpu())


@pytest.mark.parametrize("mesh,sA,sB,sC,I,J,K,flags", [
    (Y2, ((), ("Y",)), (("Y",), ()), ((), ()), 2048, 4096, 512, "FUSED"),       # 40 MB: row blocks
    (XY22, (("X",), ()), ((), ("Y",)), (("X",), ("Y",)), 512, 256, 768, "0"),  # no reduction
])
def test_run_host_fp32_cuda_cores(s, mesh, sA, sB, sC, I, J, K, flags):
    """fp32 operands run on the CUDA-core GEMM; shmm_run_host stages them the
    same way (row blocks of a fused all-reduce included), bit for bit the
    device path."""
    from partial_sum_reduction_gb300 import helpers as H
    A, B = shmm_inputs.scaled_normal_pair(I, J, K, "f32", seed=I + J)
    plan = s.Plan(mesh, sA, sB, sC, I, J, K, "f32", "f32", _flags(s, flags))
    assert plan.info.tensor_core == 0
    A_d, B_d = H.shard(plan, s.TENSOR_A, A), H.shard(plan, s.TENSOR_B, B)
    C_d = H.alloc(plan, s.TENSOR_C, fill=float("nan"))
    ws = H.workspace(plan)
    plan.run(A_d, B_d, C_d, ws)
    C_h = torch.full((I, K), float("nan")).pin_memory()
    A_r, B_r = H.alloc(plan, s.TENSOR_A), H.alloc(plan, s.TENSOR_B)
    C_r = H.alloc(plan, s.TENSOR_C, fill=float("nan"))
    plan.run_host(A.pin_memory(), B.pin_memory(), C_h, A_r, B_r, C_r, ws)
    s.shmm_sync_status()
    torch.cuda.synchronize()
    for x, y in zip(C_r, C_d):
        assert torch.equal(x, y)
    assert torch.equal(C_h, _stitch(plan, s, C_d, I, K, torch.float32))
