"""Shared helpers of the GPU parity tests: run a sharded matmul through the
C-ABI on seeded inputs and compare each rank's block with the oracle's."""
import numpy as np
import torch

import oracle

BF16_TOL = 1e-2   # max|C_gpu - C_ref| <= 1e-2 * max|C_ref| for bf16 inputs
F32P_TOL = 1e-4   # fp32 partials from bf16 products: fp32 accumulation only


def lib():
    from partial_sum_reduction_gb300 import build
    build.build()
    import partial_sum_reduction_gb300 as s
    return s


def tile_rows(n_rows, tile=256, salt=0):
    """One output row in every ``tile``-row block of [0, n_rows), at an
    offset inside the block that changes from block to block (so both
    128-row halves of a CTA pair's tile and every lane quadrant are hit over
    the blocks), plus the first and last rows."""
    rows = {0, n_rows - 1}
    for t in range((n_rows + tile - 1) // tile):
        rows.add(min(n_rows - 1, t * tile + (t * 89 + 37 * salt + 3) % tile))
    return sorted(rows)


def run_gpu(mesh, sA, sB, sC, A, B, in_dtype, out_dtype, flags=0, fill=float("nan")):
    """A, B: global CPU tensors in the input dtype.  Returns (plan, per-rank
    CPU outputs)."""
    s = lib()
    from partial_sum_reduction_gb300 import helpers as H
    I, J = A.shape
    K = B.shape[1]
    plan = s.Plan(mesh, sA, sB, sC, I, J, K, in_dtype, out_dtype, flags)
    A_r = H.shard(plan, s.TENSOR_A, A)
    B_r = H.shard(plan, s.TENSOR_B, B)
    C_r = H.alloc(plan, s.TENSOR_C, fill=fill)
    ws = H.workspace(plan)
    plan.run(A_r, B_r, C_r, ws)
    s.shmm_sync_status()
    torch.cuda.synchronize()
    return plan, [c.cpu() for c in C_r]


def oracle_run(mesh, sA, sB, sC, A, B, out_dtype, gelu=False, order="sequential", rows=None):
    return oracle.sharded_matmul(mesh, sA, sB, sC, A.float().numpy(), B.float().numpy(),
                                 out_dtype=out_dtype, gelu=gelu, order=order, rows=rows, nthreads=8)


def compare(plan, gpu, ores, exact, tol=BF16_TOL, rows=None):
    """Per rank: same box as the oracle, values equal (exact) or within
    tol * max|C_ref| over the whole result.  Returns the max abs error."""
    from partial_sum_reduction_gb300 import TENSOR_C
    ref_max = 0.0
    err = 0.0
    for r, g in enumerate(gpu):
        (o0, o1), ext = plan.rank_box(TENSOR_C, r)
        gv = g.float().numpy()
        if rows is None:
            (ro, rblk) = ores[r]
            assert (o0, o1) == tuple(ro) and tuple(ext) == rblk.shape, (r, (o0, o1), ext, ro, rblk.shape)
            ref = rblk
        else:
            crow, k0, ref = ores[r]
            assert k0 == o1
            gv = gv[np.asarray(crow, dtype=np.int64) - o0]
        assert not np.isnan(gv).any(), "rank %d: output left unwritten" % r
        if exact:
            np.testing.assert_array_equal(gv, ref, err_msg="rank %d" % r)
        if ref.size:
            ref_max = max(ref_max, float(np.abs(ref).max()))
            err = max(err, float(np.abs(gv.astype(np.float64) - ref).max()))
    if not exact:
        assert err <= tol * ref_max, "max|err| %.3g > %.1g * max|ref| %.3g" % (err, tol, ref_max)
    return err
