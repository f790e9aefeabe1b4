"""shmm_run_static_workspace: the variant of shmm_run for callers that cannot
allocate device memory (a host framework or plugin interface that passes in
only the input and output buffers, or a caller that must not call cudaMalloc
once running).  It takes its scratch from the library's fixed 64 MiB device
array instead of a caller-supplied workspace.

Each test calls the entry point through the C-ABI twice in a row and checks
both results bit for bit against shmm_run with a workspace the test
allocates.  This file sorts last so that a run stopping at its first failure
has already run every other test."""
import ctypes

import pytest
import torch

import shmm_inputs
from parity_util import lib

pytestmark = pytest.mark.gpu

CASES = [
    # unfused reduce-scatter: fp32 partials in the scratch array
    ("{Y:2}", ((), ("Y",)), (("Y",), ()), (("Y",), ()), 512, 1024, 384),
    # case 2: the all-gathered operand in the scratch array
    ("{X:2,Y:2}", ((), ("X",)), ((), ()), ((), ()), 256, 512, 264),
    # all-reduce then all-gather of the result: partials + owner blocks
    ("{X:4,Y:2}", (("X",), ("Y",)), (("Y",), ()), ((), ()), 512, 1024, 256),
]


def _ptrs(ts):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def _static_run(s, plan, A_r, B_r, C_r):
    L = s.lib()
    stream = torch.cuda.current_stream().cuda_stream
    st = L.shmm_run_static_workspace(plan.handle, _ptrs(A_r), _ptrs(B_r), _ptrs(C_r), stream)
    assert st == 0, L.shmm_last_error()
    assert L.shmm_sync_status(stream) == 0


def _inputs(s, case, seed_shift=0):
    from partial_sum_reduction_gb300 import helpers as H
    mesh, sA, sB, sC, I, J, K = case
    A, B = shmm_inputs.scaled_normal_pair(I, J, K, "bf16", seed=I + K + seed_shift)
    plan = s.Plan(mesh, sA, sB, sC, I, J, K, "bf16", "bf16")
    return plan, H.shard(plan, s.TENSOR_A, A), H.shard(plan, s.TENSOR_B, B)


@pytest.mark.parametrize("case", range(len(CASES)))
def test_static_workspace_matches_shmm_run_on_two_calls(case):
    """Both calls give shmm_run's bits exactly: the same kernels run in the
    same order on the same inputs, whatever the array held before.  Between
    the two calls another plan, on other inputs, leaves its own scratch in
    the shared array."""
    s = lib()
    from partial_sum_reduction_gb300 import helpers as H
    plan, A_r, B_r = _inputs(s, CASES[case])
    need = plan.workspace_size()
    assert 0 < need <= s.shmm.STATIC_WORKSPACE_BYTES
    ref = H.alloc(plan, s.TENSOR_C, fill=float("nan"))
    plan.run(A_r, B_r, ref, H.workspace(plan))
    torch.cuda.synchronize()
    for call in range(2):
        if call == 1:
            other, oA, oB = _inputs(s, CASES[(case + 1) % len(CASES)], seed_shift=1)
            _static_run(s, other, oA, oB, H.alloc(other, s.TENSOR_C))
        out = H.alloc(plan, s.TENSOR_C, fill=float("nan"))
        _static_run(s, plan, A_r, B_r, out)
        for r, (o, want) in enumerate(zip(out, ref)):
            assert not torch.isnan(o.float()).any(), "call %d left rank %d's output unwritten" % (call, r)
            assert torch.equal(o, want), "call %d, rank %d differs from shmm_run" % (call, r)


def test_static_workspace_rejects_plans_above_its_size():
    s = lib()
    plan = s.Plan("{X:2,Y:2}", "I,J_Y", "J_Y,K", "I_Y,K", 4096, 4096, 4096, "bf16", "bf16")
    assert plan.workspace_size() > s.shmm.STATIC_WORKSPACE_BYTES
    dummy = (ctypes.c_void_p * 4)(*([0x10000] * 4))
    L = s.lib()
    assert L.shmm_run_static_workspace(plan.handle, dummy, dummy, dummy, None) == s.shmm.ERR_NOMEM
    assert b"static workspace" in L.shmm_last_error()
