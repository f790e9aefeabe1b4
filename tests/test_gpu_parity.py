"""GPU parity: every step of the sharded matmul through the C-ABI against
the CPU oracle on the same seeded inputs -- bit-exact for integer-valued
fp32 and for the standalone reductions of given partials, within
1e-2 * max|C_ref| for bf16 products."""
import numpy as np
import pytest
import torch

import oracle
import shmm_inputs
from parity_util import BF16_TOL, F32P_TOL, compare, lib, oracle_run, run_gpu, tile_rows

pytestmark = pytest.mark.gpu

Y2 = [("Y", 2)]
XY22 = [("X", 2), ("Y", 2)]
XY42 = [("X", 4), ("Y", 2)]
X8 = [("X", 8)]


@pytest.fixture(scope="module")
def s():
    assert torch.cuda.is_available()
    return lib()


# Tensor-core GEMM variants: CTA pairs with the launcher's tile width, CTA
# pairs forced to 256 x 256 or 256 x 512 tiles, and single CTAs.
KERNELS = ["pair", "pair_narrow", "pair_wide", "single"]


def use_kernel(monkeypatch, kernel):
    monkeypatch.setenv("SHMM_TC_PAIR", "0" if kernel == "single" else "1")
    if kernel == "pair_narrow":
        monkeypatch.setenv("SHMM_TC_WIDE", "0")
    elif kernel == "pair_wide":
        monkeypatch.setenv("SHMM_TC_WIDE", "1")
    else:
        monkeypatch.delenv("SHMM_TC_WIDE", raising=False)


# ------------------------------------------------- split-K integer, {Y:2}

@pytest.mark.parametrize("flags", [0, "FUSED", "SIMT", "FUSED|SIMT", "TREE"])
@pytest.mark.parametrize("sC", [(("Y",), ()), ((), ())])
def test_split_k_integer_fp32_bit_exact(s, flags, sC):
    fl = 0
    for f in str(flags).split("|"):
        fl |= getattr(s, "FLAG_" + f) if f != "0" else 0
    A, B = shmm_inputs.split_k_integer(64, 64, 64, seed=0)
    sA, sB = ((), ("Y",)), (("Y",), ())
    plan, gpu = run_gpu(Y2, sA, sB, sC, A, B, "f32", "f32", fl)
    _, ores = oracle_run(Y2, sA, sB, sC, A, B, "f32")
    compare(plan, gpu, ores, exact=True)


def test_worked_example_on_gpu(s, golden):
    g = golden("p2_worked_example.txt")
    A = torch.tensor(g["A"], dtype=torch.float32)
    B = torch.tensor(g["B"], dtype=torch.float32)
    from partial_sum_reduction_gb300 import helpers as H
    # local partials, reduce-scatter by rows, all-gather back
    p = s.Plan("{Y:2}", "I,J_Y", "J_Y,K", "I_Y,K", 2, 2, 2, "f32", "f32")
    A_r, B_r = H.shard(p, s.TENSOR_A, A), H.shard(p, s.TENSOR_B, B)
    P_r = H.alloc(p, s.TENSOR_P, fill=float("nan"))
    p.local_matmul(A_r, B_r, P_r)
    C_r = H.alloc(p, s.TENSOR_C, fill=float("nan"))
    p.reduce_scatter(P_r, C_r)
    torch.cuda.synchronize()
    assert P_r[0].cpu().tolist() == g["partial_rank0"]
    assert P_r[1].cpu().tolist() == g["partial_rank1"]
    assert C_r[0].cpu().tolist() == g["reduce_scatter_rank0"]
    assert C_r[1].cpu().tolist() == g["reduce_scatter_rank1"]
    # all-gather of the finished rows: a plan whose result is row-owned and
    # requested whole
    pg = s.Plan("{Y:2}", "I_Y,J", "J,K", "I,K", 2, 2, 2, "f32", "f32")
    full = H.alloc(pg, s.TENSOR_C, fill=float("nan"))
    pg.all_gather(s.TENSOR_C, C_r, full)
    torch.cuda.synchronize()
    for f in full:
        assert f.cpu().tolist() == g["all_gather_every_rank"]
    # all-reduce plan end to end, fused
    pa = s.Plan("{Y:2}", "I,J_Y", "J_Y,K", "I,K", 2, 2, 2, "f32", "f32", s.FLAG_FUSED)
    Ca = H.alloc(pa, s.TENSOR_C, fill=float("nan"))
    pa.run(A_r, B_r, Ca)
    torch.cuda.synchronize()
    for c in Ca:
        assert c.cpu().tolist() == g["all_gather_every_rank"]


# --------------------------------------------- local GEMM (tensor cores)

@pytest.mark.parametrize("pair", KERNELS)
@pytest.mark.parametrize("M,Kd,N", [(128, 64, 256), (300, 200, 328), (520, 1032, 264), (7, 16, 8),
                                    (256, 4096, 512), (129, 72, 1000), (700, 136, 600)])
def test_local_gemm_partials(s, M, Kd, N, pair, monkeypatch):
    """Several tiles, ragged tails in all three dims, partial k-blocks; the
    CTA-pair kernel (256-row tiles, for M > 128) and the single-CTA kernel."""
    use_kernel(monkeypatch, pair)
    from partial_sum_reduction_gb300 import helpers as H
    A, B = shmm_inputs.scaled_normal_pair(M, 2 * Kd, N, "bf16", seed=M + N)
    p = s.Plan(Y2, ((), ("Y",)), (("Y",), ()), ((), ()), M, 2 * Kd, N, "bf16", "bf16")
    assert p.info.tensor_core == 1
    A_r, B_r = H.shard(p, s.TENSOR_A, A), H.shard(p, s.TENSOR_B, B)
    P_r = H.alloc(p, s.TENSOR_P, fill=float("nan"))
    p.local_matmul(A_r, B_r, P_r)
    s.shmm_sync_status()
    torch.cuda.synchronize()
    _, parts = oracle.partials(Y2, ((), ("Y",)), (("Y",), ()), A.float().numpy(), B.float().numpy(),
                               nthreads=8)
    for r in range(2):
        ref = parts[r][1]
        got = P_r[r].cpu().numpy()
        assert not np.isnan(got).any()
        err = np.abs(got.astype(np.float64) - ref).max()
        assert err <= F32P_TOL * np.abs(ref).max(), (r, err)


def test_tensor_core_agrees_with_cuda_cores(s):
    A, B = shmm_inputs.scaled_normal_pair(384, 512, 264, "bf16", seed=9)
    sA, sB, sC = ((), ("Y",)), (("Y",), ()), (("Y",), ())
    p1, g1 = run_gpu(Y2, sA, sB, sC, A, B, "bf16", "f32")
    p2, g2 = run_gpu(Y2, sA, sB, sC, A, B, "bf16", "f32", s.FLAG_SIMT)
    assert p1.info.tensor_core == 1 and p2.info.tensor_core == 0
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a.numpy(), b.numpy(), rtol=0, atol=1e-4 * float(b.abs().max()))


# ---------------------------------------- four-case sweep, mesh {X:2,Y:2}

FOUR = [
    (1, (("X",), ()), ((), ("Y",)), (("X",), ("Y",))),
    (2, ((), ("X",)), ((), ()), ((), ())),
    (3, ((), ("Y",)), (("Y",), ()), (("Y",), ())),
    (4, (("X",), ()), ((), ("X",)), (("X",), ())),
]


@pytest.mark.parametrize("case,sA,sB,sC", FOUR)
@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("pair", KERNELS)
def test_four_cases(s, case, sA, sB, sC, fused, pair, monkeypatch):
    use_kernel(monkeypatch, pair)
    A, B = shmm_inputs.scaled_normal_pair(512, 384, 640, "bf16", seed=case)
    plan, gpu = run_gpu(XY22, sA, sB, sC, A, B, "bf16", "bf16", s.FLAG_FUSED if fused else 0)
    assert plan.info.case_id == case
    oplan, ores = oracle_run(XY22, sA, sB, sC, A, B, "bf16")
    compare(plan, gpu, ores, exact=False)


@pytest.mark.parametrize("case,sA,sB,sC", FOUR)
def test_four_cases_full_size_sampled(s, case, sA, sB, sC):
    """I=J=K=2048, N(0,1)/sqrt(J), bf16: every output row sampled in every
    rank's block is checked against the oracle."""
    A, B = shmm_inputs.scaled_normal_pair(2048, 2048, 2048, "bf16", seed=0)
    plan, gpu = run_gpu(XY22, sA, sB, sC, A, B, "bf16", "bf16", s.FLAG_FUSED)
    rows = sorted(set(tile_rows(2048, tile=128, salt=case) + [1023, 1024]))
    _, ores = oracle_run(XY22, sA, sB, sC, A, B, "bf16", rows=rows)
    compare(plan, gpu, ores, exact=False, rows=rows)


# ------------------------------------------------------- ownership paths

@pytest.mark.parametrize("sC", [(("X", "Y"), ()), (("X",), ()), ((), ()), (("X",), ("Y",))])
@pytest.mark.parametrize("flags", [0, "FUSED", "TREE"])
def test_down_projection_layout_small(s, sC, flags):
    """A[I_X,J_Y].B[J_Y,K] on {X:4,Y:2}: all-reduce, reduce-scatter onto I
    and K, and all-gather of the result."""
    fl = 0 if flags == 0 else getattr(s, "FLAG_" + flags)
    A, B = shmm_inputs.scaled_normal_pair(1024, 1024, 512, "bf16", seed=4)
    sA, sB = (("X",), ("Y",)), (("Y",), ())
    plan, gpu = run_gpu(XY42, sA, sB, sC, A, B, "bf16", "bf16", fl)
    _, ores = oracle_run(XY42, sA, sB, sC, A, B, "bf16", order="pairwise" if flags == "TREE" else "sequential")
    compare(plan, gpu, ores, exact=False)


@pytest.mark.slow
def test_down_projection_full_size_sampled(s):
    A, B = shmm_inputs.scaled_normal_pair(8192, 28672, 8192, "bf16", seed=0)
    sA, sB, sC = (("X",), ("Y",)), (("Y",), ()), (("X",), ())
    plan, gpu = run_gpu(XY42, sA, sB, sC, A, B, "bf16", "bf16", s.FLAG_FUSED)
    # one row in every 256-row m-tile of every rank block (32 tiles), at a
    # varying offset, plus the rank-block edges
    rows = sorted(set(tile_rows(8192) + [2047, 2048, 6143, 6144]))
    _, ores = oracle_run(XY42, sA, sB, sC, A, B, "bf16", rows=rows)
    compare(plan, gpu, ores, exact=False, rows=rows)


# ------------------------------------------------- MLP column -> row pair

def _mlp(s, T, D, F, sY, fused, rows=None):
    from partial_sum_reduction_gb300 import helpers as H
    X, W1, W2 = shmm_inputs.mlp_pair(T, D, F, seed=0)
    fl = s.FLAG_FUSED if fused else 0
    p1 = s.Plan(X8, ((), ()), ((), ("X",)), ((), ("X",)), T, D, F, "bf16", "bf16", s.FLAG_GELU)
    X_r, W1_r = H.shard(p1, s.TENSOR_A, X), H.shard(p1, s.TENSOR_B, W1)
    H_r = H.alloc(p1, s.TENSOR_C, fill=float("nan"))
    p1.run(X_r, W1_r, H_r, H.workspace(p1))
    p2 = s.Plan(X8, ((), ("X",)), (("X",), ()), sY, T, F, D, "bf16", "bf16", fl)
    W2_r = H.shard(p2, s.TENSOR_B, W2)
    Y_r = H.alloc(p2, s.TENSOR_C, fill=float("nan"))
    p2.run(H_r, W2_r, Y_r, H.workspace(p2))   # H feeds the row-parallel GEMM as is
    s.shmm_sync_status()
    torch.cuda.synchronize()
    # oracle: same chain on the oracle's own H
    Xn, W1n, W2n = X.float().numpy(), W1.float().numpy(), W2.float().numpy()
    _, hres = oracle.sharded_matmul(X8, ((), ()), ((), ("X",)), ((), ("X",)), Xn, W1n, out_dtype="bf16",
                                    gelu=True, rows=rows, nthreads=8)
    Hn = np.zeros((T, F), np.float32)
    for r, v in hres.items():
        if rows is None:
            (i0, k0), blk = v
            Hn[i0:i0 + blk.shape[0], k0:k0 + blk.shape[1]] = blk
        else:
            crow, k0, blk = v
            Hn[np.asarray(crow), k0:k0 + blk.shape[1]] = blk
    _, yres = oracle.sharded_matmul(X8, ((), ("X",)), (("X",), ()), sY, Hn, W2n, out_dtype="bf16",
                                    rows=rows, nthreads=8)
    # H parity (bf16 activations)
    hmax = float(np.abs(Hn).max())
    for r in range(8):
        (i0, k0), ext = p1.rank_box(s.TENSOR_C, r)
        got = H_r[r].float().cpu().numpy()
        ref = Hn[i0:i0 + ext[0], k0:k0 + ext[1]]
        if rows is not None:
            got, ref = got[np.asarray(rows)], ref[np.asarray(rows)]
        assert np.abs(got - ref).max() <= BF16_TOL * hmax
    compare(p2, [y.cpu() for y in Y_r], yres, exact=False, rows=rows)


@pytest.mark.parametrize("sY", [((), ()), (("X",), ())])
@pytest.mark.parametrize("fused", [False, True])
def test_mlp_pair_small(s, sY, fused):
    _mlp(s, 384, 256, 1024, sY, fused)


@pytest.mark.slow
@pytest.mark.parametrize("sY", [((), ()), (("X",), ())])
def test_mlp_pair_full_size_sampled(s, sY):
    # one token row in every 256-row m-tile of both matmuls (32 tiles), at a
    # varying offset, plus the reduce-scatter block edges
    _mlp(s, 8192, 4096, 16384, sY, True, rows=sorted(set(tile_rows(8192, salt=1) + [1023, 1024])))


def test_chained_gemms_back_to_back(s, monkeypatch):
    """The MLP pair's two GEMMs, ten times in a row on one stream with
    nothing between the launches: each GEMM reads what the one before it
    wrote (H), and the next first GEMM overwrites the H the second one
    reads.  The pair kernel is a programmatic dependent launch (its set-up
    may overlap the kernel before it); its results must be those of plain
    stream order (SHMM_PDL=0, a synchronize after every launch), bit for
    bit, for every link of the chain."""
    from partial_sum_reduction_gb300 import helpers as H
    T, D, F = 512, 256, 8192
    X, W1, W2 = shmm_inputs.mlp_pair(T, D, F, seed=3)
    X2 = shmm_inputs.normal_matrix((T, D), 1.0, "bf16", seed=4)
    p1 = s.Plan(X8, ((), ()), ((), ("X",)), ((), ("X",)), T, D, F, "bf16", "bf16", s.FLAG_GELU)
    p2 = s.Plan(X8, ((), ("X",)), (("X",), ()), ((), ()), T, F, D, "bf16", "bf16", s.FLAG_FUSED)
    Xs = [H.shard(p1, s.TENSOR_A, X), H.shard(p1, s.TENSOR_A, X2)]
    W1_r, W2_r = H.shard(p1, s.TENSOR_B, W1), H.shard(p2, s.TENSOR_B, W2)
    H_r = H.alloc(p1, s.TENSOR_C, fill=float("nan"))
    ws1, ws2 = H.workspace(p1), H.workspace(p2)
    reps = 10
    outs = {}
    for pdl in ("1", "0"):
        monkeypatch.setenv("SHMM_PDL", pdl)
        Ys = [H.alloc(p2, s.TENSOR_C, fill=float("nan")) for _ in range(reps)]
        torch.cuda.synchronize()
        for i in range(reps):
            p1.run(Xs[i % 2], W1_r, H_r, ws1)
            if pdl == "0":
                torch.cuda.synchronize()
            p2.run(H_r, W2_r, Ys[i], ws2)
            if pdl == "0":
                torch.cuda.synchronize()
        s.shmm_sync_status()
        torch.cuda.synchronize()
        outs[pdl] = [[y.cpu() for y in Y] for Y in Ys]
    for i in range(reps):
        for a, b in zip(outs["1"][i], outs["0"][i]):
            assert torch.equal(a, b), i
    assert not torch.equal(outs["0"][0][0], outs["0"][1][0])  # the two inputs give different results


def test_cuda_graph_replay_matches_eager(s):
    """The path captured into a CUDA graph and replayed gives the bits of
    eager execution: the MLP pair's two GEMMs (the second a programmatic
    dependent of the first, fused all-reduce) and an unfused case-3 product
    (GEMM into partials, then the reduce-scatter kernel)."""
    from partial_sum_reduction_gb300 import helpers as H
    T, D, F = 512, 256, 8192
    X, W1, W2 = shmm_inputs.mlp_pair(T, D, F, seed=5)
    p1 = s.Plan(X8, ((), ()), ((), ("X",)), ((), ("X",)), T, D, F, "bf16", "bf16", s.FLAG_GELU)
    p2 = s.Plan(X8, ((), ("X",)), (("X",), ()), ((), ()), T, F, D, "bf16", "bf16", s.FLAG_FUSED)
    A, B = shmm_inputs.scaled_normal_pair(768, 1024, 640, "bf16", seed=6)
    p3 = s.Plan(Y2, ((), ("Y",)), (("Y",), ()), (("Y",), ()), 768, 1024, 640, "bf16", "bf16", 0)
    X_r, W1_r, W2_r = H.shard(p1, s.TENSOR_A, X), H.shard(p1, s.TENSOR_B, W1), H.shard(p2, s.TENSOR_B, W2)
    A_r, B_r = H.shard(p3, s.TENSOR_A, A), H.shard(p3, s.TENSOR_B, B)
    H_r, Y_r, C_r = H.alloc(p1, s.TENSOR_C), H.alloc(p2, s.TENSOR_C), H.alloc(p3, s.TENSOR_C)
    ws1, ws2, ws3 = H.workspace(p1), H.workspace(p2), H.workspace(p3)
    assert p3.workspace_size() > 0

    def chain():
        p1.run(X_r, W1_r, H_r, ws1)
        p2.run(H_r, W2_r, Y_r, ws2)
        p3.run(A_r, B_r, C_r, ws3)

    chain()
    s.shmm_sync_status()
    torch.cuda.synchronize()
    eager = [t.clone() for t in H_r + Y_r + C_r]
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        chain()  # warm the capture stream once, outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        chain()
    for _ in range(3):
        for t in H_r + Y_r + C_r:
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        s.shmm_sync_status()
        for a, b in zip(eager, H_r + Y_r + C_r):
            assert torch.equal(a, b)


@pytest.mark.parametrize("case", ["gelu_ragged", "fused_all_reduce", "fused_reduce_scatter",
                                  "case2_in_place", "case4_in_place"])
def test_half_tile_tail_keeps_the_bits(s, case, monkeypatch):
    """96 (or 256) tiles of 256x512 on 76 CTA pairs leave a last wave of 20
    (or 28) tiles, which the launcher runs as 40 (56) half tiles of 256
    columns.  A half tile adds its products in the whole tile's order, so
    every output has the bits of the launch without the split
    (SHMM_TC_HALF_TAIL=0): GeLU with a ragged last column tile, a fused
    all-reduce and reduce-scatter over 8 ranks (the accumulating mode), and
    operands read in place from their owners' shards (cases 2 and 4 on
    {X:2,Y:2}; a half tile's B boxes are looked up by their own columns)."""
    monkeypatch.setenv("SHMM_TC_PAIR", "1")
    monkeypatch.setenv("SHMM_TC_WIDE", "1")
    mesh = X8
    if case == "gelu_ragged":   # 8 ranks x 6 x 2 tiles
        spec = (((), ()), ((), ("X",)), ((), ("X",)))
        I, J, K, fl = 1536, 256, 8 * 1000, s.FLAG_GELU
    elif case in ("fused_all_reduce", "fused_reduce_scatter"):  # one group of 8: 16 x 6 tiles
        sC = ((), ()) if case == "fused_all_reduce" else (("X",), ())
        spec = (((), ("X",)), (("X",), ()), sC)
        I, J, K, fl = 4096, 8 * 128, 3072, s.FLAG_FUSED
    elif case == "case2_in_place":  # A gathered over X in place: 4 ranks x 6 x 4 tiles
        mesh, spec = XY22, (((), ("X",)), ((), ()), ((), ()))
        I, J, K, fl = 1536, 512, 2048, s.FLAG_FUSED
    else:                           # B gathered over X in place: 4 ranks x 8 x 8 tiles
        mesh, spec = XY22, ((("X",), ()), ((), ("X",)), (("X",), ()))
        I, J, K, fl = 4096, 512, 4096, s.FLAG_FUSED
    A, B = shmm_inputs.scaled_normal_pair(I, J, K, "bf16", seed=80)
    outs = []
    for split in ("1", "0"):
        monkeypatch.setenv("SHMM_TC_HALF_TAIL", split)
        p, g = run_gpu(mesh, *spec, A, B, "bf16", "bf16", fl)
        outs.append(g)
    if case.endswith("in_place"):
        assert p.info.fused_gather == 1
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    rows = sorted(set(tile_rows(I, salt=5)))
    _, ores = oracle_run(mesh, *spec, A, B, "bf16", gelu=case == "gelu_ragged", rows=rows)
    compare(p, outs[0], ores, exact=False, rows=rows)


# -------------------------------------------- collectives on given partials

@pytest.mark.parametrize("G", [2, 3, 4, 5, 8, 12, 16, 24, 32])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("order", ["sequential", "pairwise"])
@pytest.mark.parametrize("numel", [1 << 16, 4099 * 8])
def test_collectives_bit_exact(s, G, dtype, order, numel):
    """Reduce-scatter, all-reduce and all-gather of given partial buffers
    ({X:G}), bit for bit against the oracle in the same order.  G = 24 and
    32 take the runtime-G sequential kernel and the 32-lane shuffle tree."""
    from partial_sum_reduction_gb300 import helpers as H
    cols = 64 if numel % (64 * G) == 0 else 8
    rows = numel // cols
    if rows % G:
        rows -= rows % G
    bufs = [b[:rows * cols].reshape(rows, cols) for b in shmm_inputs.partial_buffers(G, numel, dtype, seed=G)]
    fl = s.FLAG_PARTIAL_OUT_DTYPE | (s.FLAG_TREE if order == "pairwise" else 0)
    mesh = [("X", G)]
    p_rs = s.Plan(mesh, ((), ("X",)), (("X",), ()), (("X",), ()), rows, G, cols, dtype, dtype, fl)
    p_ar = s.Plan(mesh, ((), ("X",)), (("X",), ()), ((), ()), rows, G, cols, dtype, dtype, fl)
    P_r = [b.cuda() for b in bufs]
    rs = H.alloc(p_rs, s.TENSOR_C, fill=float("nan"))
    ar = H.alloc(p_ar, s.TENSOR_C, fill=float("nan"))
    p_rs.reduce_scatter(P_r, rs)
    p_ar.all_reduce(P_r, ar)
    pg = s.Plan(mesh, (("X",), ()), ((), ()), ((), ()), rows, 8, cols, dtype, dtype)
    ag = H.alloc(pg, s.TENSOR_C, fill=float("nan"))
    pg.all_gather(s.TENSOR_C, rs, ag)
    torch.cuda.synchronize()
    ref_rs = oracle.collective_reduce([b.float().numpy() for b in bufs], "reduce_scatter", dtype, order=order)
    ref_ar = oracle.collective_reduce([b.float().numpy() for b in bufs], "all_reduce", dtype, order=order)
    for q in range(G):
        np.testing.assert_array_equal(rs[q].float().cpu().numpy(), ref_rs[q])
        np.testing.assert_array_equal(ar[q].float().cpu().numpy(), ref_ar[q])
        # AllReduce = ReduceScatter + AllGather, bit for bit
        np.testing.assert_array_equal(ag[q].float().cpu().numpy(), ref_ar[q])


@pytest.mark.parametrize("G", [2, 3, 4])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("order", ["sequential", "pairwise"])
def test_collectives_scalar_path(s, G, dtype, order):
    """Owner blocks that are not whole 16-byte vectors (odd row width)."""
    from partial_sum_reduction_gb300 import helpers as H
    rows, cols = 12, 5
    bufs = [b.reshape(rows, cols) for b in shmm_inputs.partial_buffers(G, rows * cols, dtype, seed=7)]
    fl = s.FLAG_PARTIAL_OUT_DTYPE | (s.FLAG_TREE if order == "pairwise" else 0)
    mesh = [("X", G)]
    p = s.Plan(mesh, ((), ("X",)), (("X",), ()), (("X",), ()), rows, G, cols, dtype, dtype, fl)
    pa = s.Plan(mesh, ((), ("X",)), (("X",), ()), ((), ()), rows, G, cols, dtype, dtype, fl)
    rs = H.alloc(p, s.TENSOR_C, fill=float("nan"))
    ar = H.alloc(pa, s.TENSOR_C, fill=float("nan"))
    P_r = [b.cuda() for b in bufs]
    p.reduce_scatter(P_r, rs)
    pa.all_reduce(P_r, ar)
    torch.cuda.synchronize()
    host = [b.float().numpy() for b in bufs]
    ref_rs = oracle.collective_reduce(host, "reduce_scatter", dtype, order=order)
    ref_ar = oracle.collective_reduce(host, "all_reduce", dtype, order=order)
    for q in range(G):
        np.testing.assert_array_equal(rs[q].float().cpu().numpy(), ref_rs[q])
        np.testing.assert_array_equal(ar[q].float().cpu().numpy(), ref_ar[q])


def _bits_equal(got, ref, what):
    """Bit-for-bit equality of fp32 arrays (so +0 and -0 differ too)."""
    g = np.ascontiguousarray(got, dtype=np.float32).view(np.uint32)
    r = np.ascontiguousarray(ref, dtype=np.float32).view(np.uint32)
    assert g.shape == r.shape, what
    bad = np.flatnonzero(g.ravel() != r.ravel())
    assert bad.size == 0, "%s: %d elements differ, first at %d" % (what, bad.size, bad[0])


@pytest.mark.slow
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_collectives_at_one_gib_per_rank(s, dtype):
    """Two ranks with 1 GiB partial buffers each, the largest size of the
    collective sweep, through the same launchers and grids the benchmark
    times: reduce-scatter over rows, all-reduce, and the all-gather of the
    owner blocks, bit for bit against the oracle's sequential rank sum."""
    from partial_sum_reduction_gb300 import helpers as H
    G, eb = 2, (4 if dtype == "f32" else 2)
    numel = (1 << 30) // eb
    cols = 4096
    rows = numel // cols
    bufs = [b.reshape(rows, cols) for b in shmm_inputs.partial_buffers(G, numel, dtype, seed=30)]
    mesh = [("X", G)]
    fl = s.FLAG_PARTIAL_OUT_DTYPE
    p_rs = s.Plan(mesh, ((), ("X",)), (("X",), ()), (("X",), ()), rows, G, cols, dtype, dtype, fl)
    p_ar = s.Plan(mesh, ((), ("X",)), (("X",), ()), ((), ()), rows, G, cols, dtype, dtype, fl)
    pg = s.Plan(mesh, (("X",), ()), ((), ()), ((), ()), rows, 8, cols, dtype, dtype)
    P_r = [b.cuda() for b in bufs]
    rs = H.alloc(p_rs, s.TENSOR_C, fill=float("nan"))
    p_rs.reduce_scatter(P_r, rs)
    ar = H.alloc(p_ar, s.TENSOR_C, fill=float("nan"))
    p_ar.all_reduce(P_r, ar)
    ag = H.alloc(pg, s.TENSOR_C, fill=float("nan"))
    pg.all_gather(s.TENSOR_C, rs, ag)
    s.shmm_sync_status()
    torch.cuda.synchronize()
    del P_r
    host = [b.float().numpy() for b in bufs]
    del bufs
    ref = oracle.collective_reduce(host, "reduce_scatter", dtype)
    for q in range(G):
        _bits_equal(rs[q].float().cpu().numpy(), ref[q], "reduce-scatter owner %d" % q)
    del ref
    ref = oracle.collective_reduce(host, "all_reduce", dtype)[0]
    for q in range(G):
        _bits_equal(ar[q].float().cpu().numpy(), ref, "all-reduce member %d" % q)
        _bits_equal(ag[q].float().cpu().numpy(), ref, "all-gather member %d" % q)


@pytest.mark.slow
@pytest.mark.parametrize("dtype,order", [("f32", "sequential"), ("bf16", "sequential"), ("f32", "pairwise")])
def test_collectives_eight_ranks_at_256_mib(s, dtype, order):
    """Eight ranks of 256 MiB partials: the reduce-scatter bench.py times
    beside every benchmark line (fp32, rank order), with the grid and
    unrolling of the eight-rank kernels, bit for bit against the oracle."""
    from partial_sum_reduction_gb300 import helpers as H
    G, eb = 8, (4 if dtype == "f32" else 2)
    numel = (256 << 20) // eb
    cols = 4096
    rows = numel // cols
    bufs = [b.reshape(rows, cols) for b in shmm_inputs.partial_buffers(G, numel, dtype, seed=31)]
    mesh = [("X", G)]
    fl = s.FLAG_PARTIAL_OUT_DTYPE | (s.FLAG_TREE if order == "pairwise" else 0)
    p_rs = s.Plan(mesh, ((), ("X",)), (("X",), ()), (("X",), ()), rows, G, cols, dtype, dtype, fl)
    p_ar = s.Plan(mesh, ((), ("X",)), (("X",), ()), ((), ()), rows, G, cols, dtype, dtype, fl)
    P_r = [b.cuda() for b in bufs]
    rs = H.alloc(p_rs, s.TENSOR_C, fill=float("nan"))
    p_rs.reduce_scatter(P_r, rs)
    ar = H.alloc(p_ar, s.TENSOR_C, fill=float("nan"))
    p_ar.all_reduce(P_r, ar)
    s.shmm_sync_status()
    torch.cuda.synchronize()
    del P_r
    host = [b.float().numpy() for b in bufs]
    del bufs
    ref = oracle.collective_reduce(host, "reduce_scatter", dtype, order=order)
    for q in range(G):
        _bits_equal(rs[q].float().cpu().numpy(), ref[q], "reduce-scatter owner %d" % q)
    del ref
    ref = oracle.collective_reduce(host, "all_reduce", dtype, order=order)[0]
    for q in range(G):
        _bits_equal(ar[q].float().cpu().numpy(), ref, "all-reduce member %d" % q)


@pytest.mark.parametrize("G", [2, 4])
def test_reduce_scatter_onto_columns(s, G):
    from partial_sum_reduction_gb300 import helpers as H
    rows, cols = 96, 40 * G
    bufs = [b.reshape(rows, cols) for b in shmm_inputs.partial_buffers(G, rows * cols, "f32", seed=3)]
    mesh = [("X", G)]
    p = s.Plan(mesh, ((), ("X",)), (("X",), ()), ((), ("X",)), rows, G, cols, "f32", "bf16")
    out = H.alloc(p, s.TENSOR_C, fill=float("nan"))
    p.reduce_scatter([b.cuda() for b in bufs], out)
    torch.cuda.synchronize()
    ref = oracle.collective_reduce([b.numpy() for b in bufs], "reduce_scatter", "bf16", scatter_dim=1)
    for q in range(G):
        np.testing.assert_array_equal(out[q].float().cpu().numpy(), ref[q])


def test_operand_all_gather_bit_exact(s):
    from partial_sum_reduction_gb300 import helpers as H
    A, B = shmm_inputs.scaled_normal_pair(256, 512, 264, "bf16", seed=1)
    # case 2 gathers A along J; case 4 gathers B along K
    cases = [(((), ("X",)), ((), ()), s.TENSOR_A, s.TENSOR_A_LOCAL, A),
             ((("X",), ()), ((), ("X",)), s.TENSOR_B, s.TENSOR_B_LOCAL, B)]
    for sA, sB, t, tloc, full in cases:
        p = s.Plan(XY22, sA, sB, ((), ()), 256, 512, 264, "bf16", "bf16")
        shards = H.shard(p, t, full)
        loc = H.alloc(p, tloc)
        p.all_gather(t, shards, loc)
        torch.cuda.synchronize()
        for r in range(4):
            (o0, o1), ext = p.rank_box(tloc, r)
            assert torch.equal(loc[r].cpu(), full[o0:o0 + ext[0], o1:o1 + ext[1]])


# -------------------------------------------------------------- invariants

@pytest.mark.parametrize("pair", KERNELS)
def test_fused_equals_unfused_bitwise(s, pair, monkeypatch):
    """SHMM_FLAG_RANK_ORDER: the fused epilogue adds per-rank partials in
    ascending rank order, exactly the standalone sequential reduction."""
    use_kernel(monkeypatch, pair)
    A, B = shmm_inputs.scaled_normal_pair(640, 1024, 512, "bf16", seed=12)
    for mesh, sA, sB, sC in ((Y2, ((), ("Y",)), (("Y",), ()), (("Y",), ())),
                             (XY42, (("X",), ("Y",)), (("Y",), ()), (("X",), ())),
                             ([("X", 4)], ((), ("X",)), (("X",), ()), ((), ("X",)))):
        _, g1 = run_gpu(mesh, sA, sB, sC, A, B, "bf16", "f32")
        p2, g2 = run_gpu(mesh, sA, sB, sC, A, B, "bf16", "f32", s.FLAG_FUSED | s.FLAG_RANK_ORDER)
        assert p2.info.fused == 1
        for a, b in zip(g1, g2):
            assert torch.equal(a, b)


@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("pair", KERNELS)
def test_gelu_after_the_reduction_fused_equals_unfused(s, pair, out, monkeypatch):
    """GeLU of a reduced sum: applied by the standalone reduction kernel,
    or by the GEMM epilogue after the rank-order fold.  Same sums, same
    GeLU, so the same bits.  Pre-activations span about +-20: both tails
    and the zero crossing."""
    use_kernel(monkeypatch, pair)
    A = shmm_inputs.normal_matrix((640, 1024), 1.0, "bf16", seed=14)
    B = shmm_inputs.normal_matrix((1024, 512), 4.0 / 1024 ** 0.5, "bf16", seed=15)
    for mesh, sA, sB, sC in ((Y2, ((), ("Y",)), (("Y",), ()), (("Y",), ())),
                             ([("X", 4)], ((), ("X",)), (("X",), ()), ((), ("X",)))):
        _, g1 = run_gpu(mesh, sA, sB, sC, A, B, "bf16", out, s.FLAG_GELU)
        p2, g2 = run_gpu(mesh, sA, sB, sC, A, B, "bf16", out, s.FLAG_GELU | s.FLAG_FUSED | s.FLAG_RANK_ORDER)
        assert p2.info.fused == 1
        assert min(float(c.float().min()) for c in g1) < -0.1 and max(float(c.float().max()) for c in g1) > 8.0
        for a, b in zip(g1, g2):
            assert torch.equal(a, b)


@pytest.mark.parametrize("pair", KERNELS)
def test_accumulating_fusion_is_one_contraction(s, pair, monkeypatch):
    """Default fused path: a reduction group's products accumulate in one
    fp32 accumulator, k-block after k-block in ascending rank order -- the
    same tensor-core operations as one unsharded GEMM over the whole J, so
    every output element has the same bits (J_r a multiple of the 64-wide
    k-block, so block edges coincide)."""
    use_kernel(monkeypatch, pair)
    A, B = shmm_inputs.scaled_normal_pair(640, 1024, 512, "bf16", seed=13)
    _, full = run_gpu([("Y", 1)], ((), ()), ((), ()), ((), ()), A, B, "bf16", "f32")
    full = full[0]
    for mesh, sA, sB, sC in ((Y2, ((), ("Y",)), (("Y",), ()), (("Y",), ())),
                             (XY42, (("X",), ("Y",)), (("Y",), ()), (("X",), ())),
                             (X8, ((), ("X",)), (("X",), ()), ((), ())),
                             ([("X", 4)], ((), ("X",)), (("X",), ()), ((), ("X",)))):
        p, g = run_gpu(mesh, sA, sB, sC, A, B, "bf16", "f32", s.FLAG_FUSED)
        assert p.info.fused == 1
        for r, c in enumerate(g):
            (o0, o1), ext = p.rank_box(s.TENSOR_C, r)
            assert torch.equal(c, full[o0:o0 + ext[0], o1:o1 + ext[1]]), (mesh, r)


@pytest.mark.parametrize("flags", ["FUSED", "FUSED|RANK_ORDER", "0"])
@pytest.mark.parametrize("sC", [((), ()), (("X",), ()), ((), ("X",))])
def test_integer_bf16_tensor_core_bit_exact(s, flags, sC):
    """Integer-valued bf16 operands on the tensor cores, {X:8}: every
    partial and every sum is an integer below 2^24, so all reduction orders
    give the oracle's exact result."""
    fl = 0
    for f in flags.split("|"):
        fl |= getattr(s, "FLAG_" + f) if f != "0" else 0
    A, B = shmm_inputs.split_k_integer(384, 1024, 320, seed=4)
    A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    sA, sB = ((), ("X",)), (("X",), ())
    plan, gpu = run_gpu(X8, sA, sB, sC, A, B, "bf16", "f32", fl)
    assert plan.info.tensor_core == 1
    _, ores = oracle_run(X8, sA, sB, sC, A, B, "f32")
    compare(plan, gpu, ores, exact=True)


# ------------------------------------------- 256 x 512 tiles on CTA pairs

WIDE = [
    # name, mesh, sA, sB, sC, I, J, K, flags, out dtype
    ("case1_two_tiles", XY22, (("X",), ()), ((), ("Y",)), (("X",), ("Y",)), 768, 512, 1536, "0", "bf16"),
    ("gelu_ragged_n", X8, ((), ()), ((), ("X",)), ((), ("X",)), 512, 256, 8 * 640, "GELU", "bf16"),
    ("fused_all_reduce", XY42, (("X",), ("Y",)), (("Y",), ()), (("X",), ()), 1024, 1024, 1280, "FUSED", "bf16"),
    ("fused_rs_rows", X8, ((), ("X",)), (("X",), ()), (("X",), ()), 2048, 1024, 1024, "FUSED", "f32"),
    ("fused_rs_cols", [("X", 4)], ((), ("X",)), (("X",), ()), ((), ("X",)), 512, 512, 2048, "FUSED", "bf16"),
    # owner blocks of 260 rows: per-thread stores instead of bulk tensor stores
    ("fused_rs_rows_per_thread", [("X", 2)], ((), ("X",)), (("X",), ()), (("X",), ()), 520, 256, 1032, "FUSED",
     "f32"),
    ("in_place_gather_b", XY22, (("X",), ()), ((), ("X",)), (("X",), ()), 512, 384, 1280, "FUSED", "f32"),
    ("ragged_m", Y2, ((), ("Y",)), (("Y",), ()), ((), ()), 300, 256, 1000, "FUSED", "bf16"),
]


@pytest.mark.parametrize("name,mesh,sA,sB,sC,I,J,K,flags,out", WIDE, ids=[w[0] for w in WIDE])
def test_wide_tiles_equal_narrow_bitwise(s, name, mesh, sA, sB, sC, I, J, K, flags, out, monkeypatch):
    """256 x 512 tiles (two MMAs per K step sharing the A operand, one tile
    filling TMEM) add every output element's products over the same
    k-blocks in the same order as 256 x 256 tiles, so both give the same
    bits in every write mode; and both match the oracle."""
    fl = 0
    for f in flags.split("|"):
        fl |= getattr(s, "FLAG_" + f) if f != "0" else 0
    A, B = shmm_inputs.scaled_normal_pair(I, J, K, "bf16", seed=I + K)
    monkeypatch.setenv("SHMM_TC_WIDE", "0")
    _, g1 = run_gpu(mesh, sA, sB, sC, A, B, "bf16", out, fl)
    monkeypatch.setenv("SHMM_TC_WIDE", "1")
    p2, g2 = run_gpu(mesh, sA, sB, sC, A, B, "bf16", out, fl)
    assert p2.info.tensor_core == 1 and p2.info.local_I > 128
    for a, b in zip(g1, g2):
        assert torch.equal(a, b), name
    _, ores = oracle_run(mesh, sA, sB, sC, A, B, out, gelu="GELU" in flags)
    compare(p2, g2, ores, exact=False, tol=BF16_TOL if out == "bf16" else F32P_TOL)


def test_all_reduce_replicas_identical(s):
    A, B = shmm_inputs.scaled_normal_pair(256, 2048, 384, "bf16", seed=2)
    plan, gpu = run_gpu(X8, ((), ("X",)), (("X",), ()), ((), ()), A, B, "bf16", "bf16", s.FLAG_FUSED)
    for g in gpu[1:]:
        assert torch.equal(g, gpu[0])


# -------------------------------------------------------------- edge cases

@pytest.mark.parametrize("dtype,flags", [("f32", 0), ("bf16", 0), ("bf16", "FUSED"), ("bf16", "GELU")])
def test_empty_contraction_gives_zero(s, dtype, flags):
    """J = 0: every output element is the empty sum, 0 (GeLU(0) = 0), on
    every path the plan can take, fused or not; nothing is left unwritten."""
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    fl = {0: 0, "FUSED": s.FLAG_FUSED, "GELU": s.FLAG_GELU}[flags]
    A = torch.zeros(64, 0, dtype=tdt)
    B = torch.zeros(0, 32, dtype=tdt)
    plan, gpu = run_gpu(Y2, ((), ("Y",)), (("Y",), ()), (("Y",), ()), A, B, dtype, dtype, fl)
    for g in gpu:
        assert torch.equal(g, torch.zeros_like(g))


def test_empty_output_is_a_no_op(s):
    A = torch.ones(0, 16, dtype=torch.bfloat16)
    B = torch.ones(16, 8, dtype=torch.bfloat16)
    plan, gpu = run_gpu(Y2, ((), ("Y",)), (("Y",), ()), ((), ()), A, B, "bf16", "bf16")
    assert all(g.numel() == 0 for g in gpu)


@pytest.mark.parametrize("I,J,K", [(1, 2, 1), (3, 6, 5), (17, 10, 9), (130, 14, 70)])
def test_ragged_shapes_off_the_tensor_core_path(s, I, J, K):
    A, B = shmm_inputs.scaled_normal_pair(I, J, K, "bf16", seed=I)
    plan, gpu = run_gpu(Y2, ((), ("Y",)), (("Y",), ()), ((), ()), A, B, "bf16", "bf16", s.FLAG_FUSED)
    _, ores = oracle_run(Y2, ((), ("Y",)), (("Y",), ()), ((), ()), A, B, "bf16")
    compare(plan, gpu, ores, exact=False)


def test_outputs_stay_inside_their_boxes(s):
    """Canary-filled guard regions around every rank's output slice of one
    allocation stay untouched."""
    from partial_sum_reduction_gb300 import helpers as H
    A, B = shmm_inputs.scaled_normal_pair(384, 512, 200, "bf16", seed=5)
    for flags in (0, s.FLAG_FUSED):
        p = s.Plan(XY42, (("X",), ("Y",)), (("Y",), ()), (("X", "Y"), ()), 384, 512, 200, "bf16", "bf16",
                   flags)
        A_r, B_r = H.shard(p, s.TENSOR_A, A), H.shard(p, s.TENSOR_B, B)
        _, ext = p.rank_box(s.TENSOR_C, 0)
        n = ext[0] * ext[1]
        guard = 4096
        pool = torch.full((8 * (n + 2 * guard),), -7.0, dtype=torch.bfloat16, device="cuda")
        C_r = [pool[r * (n + 2 * guard) + guard: r * (n + 2 * guard) + guard + n].view(ext) for r in range(8)]
        p.run(A_r, B_r, C_r, H.workspace(p))
        torch.cuda.synchronize()
        host = pool.cpu()
        for r in range(8):
            base = r * (n + 2 * guard)
            assert torch.all(host[base:base + guard] == -7.0)
            assert torch.all(host[base + guard + n:base + 2 * guard + n] == -7.0)


# ------------------------------------------------------- failure detection

def test_bounded_wait_reports_timeout_and_context_survives(s):
    """A wait that runs out (a barrier nothing arrives at, ~10 ms limit) is
    reported through the device status word; the next read is clean and the
    context still computes correctly."""
    s.shmm_sync_status()
    s.shmm_selftest_wait_timeout(20_000_000)
    with pytest.raises(s.ShmmError) as e:
        s.shmm_sync_status()
    assert e.value.status == s.shmm.ERR_TIMEOUT
    s.shmm_sync_status()  # cleared
    A, B = shmm_inputs.split_k_integer(64, 64, 64, seed=1)
    plan, gpu = run_gpu(Y2, ((), ("Y",)), (("Y",), ()), (("Y",), ()), A, B, "f32", "f32", s.FLAG_FUSED)
    _, ores = oracle_run(Y2, ((), ("Y",)), (("Y",), ()), (("Y",), ()), A, B, "f32")
    compare(plan, gpu, ores, exact=True)


# ------------------------------------------ in-place operand gather (f1)

GATHERS = [
    ("case2", XY22, ((), ("X",)), ((), ()), ((), ()), 384, 512, 264),
    ("case4", XY22, (("X",), ()), ((), ("X",)), (("X",), ()), 512, 384, 640),
    ("case3+4", XY22, (("X",), ("Y",)), (("Y",), ("X",)), (("X",), ()), 512, 512, 512),
    ("case2_both", XY22, ((), ("X",)), (("Y",), ()), ((), ()), 384, 512, 264),
]


@pytest.mark.parametrize("name,mesh,sA,sB,sC,I,J,K", GATHERS)
@pytest.mark.parametrize("pair", KERNELS)
def test_in_place_gather_equals_explicit_gather(s, name, mesh, sA, sB, sC, I, J, K, pair, monkeypatch):
    """Operands read from their owners' shards inside the GEMM give the same
    bits as all-gathering them first, and match the oracle."""
    use_kernel(monkeypatch, pair)
    A, B = shmm_inputs.scaled_normal_pair(I, J, K, "bf16", seed=I + J)
    p1, g1 = run_gpu(mesh, sA, sB, sC, A, B, "bf16", "f32", 0)
    p2, g2 = run_gpu(mesh, sA, sB, sC, A, B, "bf16", "f32", s.FLAG_FUSED | s.FLAG_RANK_ORDER)
    assert p1.info.fused_gather == 0 and p2.info.fused_gather == 1 and p2.workspace_size() == 0
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
    _, ores = oracle_run(mesh, sA, sB, sC, A, B, "f32")
    compare(p2, g2, ores, exact=False, tol=F32P_TOL)
    p3, g3 = run_gpu(mesh, sA, sB, sC, A, B, "bf16", "f32", s.FLAG_FUSED)  # accumulating
    assert p3.info.fused_gather == 1
    compare(p3, g3, ores, exact=False, tol=F32P_TOL)


def test_gather_falls_back_when_shards_straddle_boxes(s):
    A, B = shmm_inputs.scaled_normal_pair(256, 192, 136, "bf16", seed=3)  # shard width 96
    plan, gpu = run_gpu(XY22, ((), ("X",)), ((), ()), ((), ()), A, B, "bf16", "bf16", s.FLAG_FUSED)
    assert plan.info.fused_gather == 0
    _, ores = oracle_run(XY22, ((), ("X",)), ((), ()), ((), ()), A, B, "bf16")
    compare(plan, gpu, ores, exact=False)


# ------------------------------------------------------ all-to-all (f2)

RESHARDS = [
    ([("X", 2)], ((), ("X",)), (("X",), ())),              # A[I,J_X] -> A[I_X,J]
    ([("X", 4)], ((), ("X",)), (("X",), ())),
    ([("X", 8)], (("X",), ()), ((), ("X",))),
    ([("X", 2), ("Y", 2)], (("X",), ("Y",)), (("Y",), ("X",))),
    ([("X", 2), ("Y", 2)], ((), ("Y",)), (("X", "Y"), ())),  # replicated over X
    ([("X", 2), ("Y", 2)], (("X", "Y"), ()), ((), ())),      # all-gather as a reshard
    ([("X", 2), ("Y", 2)], ((), ()), (("Y",), ("X",))),      # slicing a replica
]


@pytest.mark.parametrize("mesh,sf,st", RESHARDS)
@pytest.mark.parametrize("dtype,shape", [("bf16", (256, 512)), ("f32", (96, 64)), ("bf16", (24, 40))])
def test_reshard_bit_exact(s, mesh, sf, st, dtype, shape):
    import oracle as orc
    rows, cols = shape
    full = shmm_inputs.uniform_matrix(shape, -1.0, 1.0, dtype, seed=rows + cols)
    N = orc.mesh_size(mesh)
    src, host_src = [], {}
    for r in range(N):
        (i0, j0), (n0, n1) = orc.shard_box(mesh, sf, shape, r)
        blk = full[i0:i0 + n0, j0:j0 + n1].contiguous()
        host_src[r] = blk.float().numpy()
        src.append(blk.cuda())
    dst = []
    for r in range(N):
        _, (n0, n1) = orc.shard_box(mesh, st, shape, r)
        dst.append(torch.full((n0, n1), float("nan"), dtype=full.dtype, device="cuda"))
    s.shmm_reshard(mesh, sf, st, rows, cols, dtype, src, dst)
    torch.cuda.synchronize()
    ref = orc.reshard(mesh, sf, st, host_src, shape)
    for r in range(N):
        np.testing.assert_array_equal(dst[r].float().cpu().numpy(), ref[r].astype(np.float32))


@pytest.mark.slow
@pytest.mark.parametrize("G,rows,cols", [(8, 8192, 16384), (2, 16384, 32768)])
def test_all_to_all_at_sweep_sizes(s, G, rows, cols):
    """The all-to-all of the collective sweep at its large end: a 256 MiB
    bf16 array over 8 ranks and a 1 GiB one over 2, moved from row shards to
    column shards through the benchmark's launcher, bit for bit against the
    oracle's reshard."""
    import oracle as orc
    mesh, sf, st = [("X", G)], (("X",), ()), ((), ("X",))
    full = shmm_inputs.uniform_matrix((rows, cols), -1.0, 1.0, "bf16", seed=G)
    src, host_src = [], {}
    for r in range(G):
        (i0, j0), (n0, n1) = orc.shard_box(mesh, sf, (rows, cols), r)
        blk = full[i0:i0 + n0, j0:j0 + n1].contiguous()
        host_src[r] = blk.float().numpy()
        src.append(blk.cuda())
    del full
    dst = []
    for r in range(G):
        _, (n0, n1) = orc.shard_box(mesh, st, (rows, cols), r)
        dst.append(torch.full((n0, n1), float("nan"), dtype=torch.bfloat16, device="cuda"))
    s.shmm_reshard(mesh, sf, st, rows, cols, "bf16", src, dst)
    s.shmm_sync_status()
    torch.cuda.synchronize()
    del src
    ref = orc.reshard(mesh, sf, st, host_src, (rows, cols))
    del host_src
    for r in range(G):
        np.testing.assert_array_equal(dst[r].float().cpu().numpy(), ref[r].astype(np.float32))


# --------------------------------------- sequence parallelism (f4)

@pytest.mark.parametrize("rows,cols,dtype", [(64, 4096, "bf16"), (33, 1000, "f32"), (7, 12000, "bf16"),
                                             (5, 1001, "bf16"), (128, 8192, "bf16"), (3, 4096, "f32")])
def test_layernorm_rows(s, rows, cols, dtype):
    x = shmm_inputs.normal_matrix((rows, cols), 2.0, dtype, seed=rows)
    g = shmm_inputs.normal_matrix((1, cols), 1.0, "f32", seed=1)[0]
    b = shmm_inputs.normal_matrix((1, cols), 1.0, "f32", seed=2)[0]
    y = torch.full_like(x, float("nan")).cuda()
    s.shmm_layernorm(x.cuda(), g.cuda(), b.cuda(), y, eps=1e-5)
    torch.cuda.synchronize()
    ref = oracle.layernorm(x.float().numpy(), g.numpy(), b.numpy(), 1e-5, dtype)
    got = y.float().cpu().numpy()
    tol = BF16_TOL if dtype == "bf16" else 1e-4
    assert np.abs(got - ref).max() <= tol * np.abs(ref).max()


@pytest.mark.parametrize("G,brows,cols,dtype", [(2, 96, 4096, "bf16"), (4, 33, 2048, "f32"), (8, 64, 8192, "bf16"),
                                                 (2, 17, 8192, "f32"), (3, 40, 1001, "bf16")])
def test_layernorm_gather_paths_agree(s, G, brows, cols, dtype, monkeypatch):
    """LayerNorm + all-gather with rows staged through shared memory (the
    bulk-copy path, several rows in flight per CTA) and with per-thread row
    loads give the same bits: the same vectors per thread and the same block
    sums.  Odd row counts leave CTAs with uneven walks; 8192 fp32 columns
    leave room for two staged rows only; rows of 1001 columns are not whole
    16-byte vectors (the element-wise path for both settings)."""
    from partial_sum_reduction_gb300 import helpers as H
    mesh = [("X", G)]
    p = s.Plan(mesh, (("X",), ()), ((), ()), ((), ()), G * brows, 8, cols, dtype, dtype)
    x = shmm_inputs.normal_matrix((G * brows, cols), 2.0, dtype, seed=G + brows)
    shards = [x[q * brows:(q + 1) * brows].contiguous().cuda() for q in range(G)]
    gamma = shmm_inputs.normal_matrix((1, cols), 1.0, "f32", seed=3)[0].cuda()
    beta = shmm_inputs.normal_matrix((1, cols), 1.0, "f32", seed=4)[0].cuda()
    outs = {}
    for bulk in ("1", "0"):
        monkeypatch.setenv("SHMM_LN_BULK", bulk)
        out = H.alloc(p, s.TENSOR_C, fill=float("nan"))
        p.layernorm_all_gather(shards, gamma, beta, out)
        s.shmm_sync_status()
        torch.cuda.synchronize()
        outs[bulk] = out
    ref = oracle.layernorm(x.float().numpy(), gamma.cpu().numpy(), beta.cpu().numpy(), 1e-5, dtype)
    tol = BF16_TOL if dtype == "bf16" else 1e-4
    for a, b in zip(outs["1"], outs["0"]):
        assert torch.equal(a, b)
        got = a.float().cpu().numpy()
        assert np.abs(got - ref).max() <= tol * np.abs(ref).max()


@pytest.mark.slow
def test_layernorm_all_gather_full_size_sampled(s, monkeypatch):
    """LayerNorm + all-gather at the sequence-parallel block's size: 8 ranks
    x 1024 token rows x 4096 bf16 columns (64 MB in, 8 copies of 64 MB out).
    Every copy holds every rank's normalised rows; one row in every 64 of
    each copy is checked against the oracle, and the bulk-copy and register
    paths agree bit for bit on all of it."""
    from partial_sum_reduction_gb300 import helpers as H
    G, brows, cols = 8, 1024, 4096
    p = s.Plan(X8, (("X",), ()), ((), ()), ((), ()), G * brows, 8, cols, "bf16", "bf16")
    x = shmm_inputs.normal_matrix((G * brows, cols), 2.0, "bf16", seed=21)
    shards = [x[q * brows:(q + 1) * brows].contiguous().cuda() for q in range(G)]
    gamma = (1.0 + 0.1 * shmm_inputs.normal_matrix((1, cols), 1.0, "f32", seed=22)[0]).cuda()
    beta = (0.1 * shmm_inputs.normal_matrix((1, cols), 1.0, "f32", seed=23)[0]).cuda()
    outs = {}
    for bulk in ("1", "0"):
        monkeypatch.setenv("SHMM_LN_BULK", bulk)
        out = H.alloc(p, s.TENSOR_C, fill=float("nan"))
        p.layernorm_all_gather(shards, gamma, beta, out)
        s.shmm_sync_status()
        torch.cuda.synchronize()
        outs[bulk] = out
    for a, b in zip(outs["1"], outs["0"]):
        assert torch.equal(a, b)
    rows = sorted(set(list(range(0, G * brows, 64)) + [q * brows - 1 for q in range(1, G + 1)]))
    ref = oracle.layernorm(x[rows].float().numpy(), gamma.cpu().numpy(), beta.cpu().numpy(), 1e-5, "bf16")
    for copy in outs["1"]:
        got = copy[rows].float().cpu().numpy()
        assert np.abs(got - ref).max() <= BF16_TOL * np.abs(ref).max()


@pytest.mark.parametrize("fused", [True, False])
def test_sequence_parallel_mlp_block(s, fused):
    """X -> GeLU(X.W1) (column-parallel) -> .W2 reduce-scattered over tokens
    -> LayerNorm per token -> all-gather, on {X:8}; equals the oracle chain,
    and (AllReduce = ReduceScatter + AllGather) equals LayerNorm applied to
    the all-reduced result bit for bit."""
    from partial_sum_reduction_gb300 import helpers as H
    T, D, F = 512, 1024, 2048
    X, W1, W2 = shmm_inputs.mlp_pair(T, D, F, seed=3)
    gam = (1.0 + 0.1 * shmm_inputs.normal_matrix((1, D), 1.0, "f32", seed=4)[0]).cuda()
    bet = (0.1 * shmm_inputs.normal_matrix((1, D), 1.0, "f32", seed=5)[0]).cuda()
    fl = s.FLAG_FUSED if fused else 0
    p1 = s.Plan(X8, ((), ()), ((), ("X",)), ((), ("X",)), T, D, F, "bf16", "bf16", s.FLAG_GELU)
    H_r = H.alloc(p1, s.TENSOR_C)
    p1.run(H.shard(p1, s.TENSOR_A, X), H.shard(p1, s.TENSOR_B, W1), H_r, H.workspace(p1))
    p2 = s.Plan(X8, ((), ("X",)), (("X",), ()), (("X",), ()), T, F, D, "bf16", "bf16", fl)
    W2_r = H.shard(p2, s.TENSOR_B, W2)
    Y_rs = H.alloc(p2, s.TENSOR_C)
    p2.run(H_r, W2_r, Y_rs, H.workspace(p2))
    pg = s.Plan(X8, (("X",), ()), ((), ()), ((), ()), T, 8, D, "bf16", "bf16")  # rows gathered over X
    Y_n = H.alloc(pg, s.TENSOR_C, fill=float("nan"))
    pg.layernorm_all_gather(Y_rs, gam, bet, Y_n, eps=1e-5)
    # the all-reduce route: full Y on every rank, normalised in place
    pa = s.Plan(X8, ((), ("X",)), (("X",), ()), ((), ()), T, F, D, "bf16", "bf16", fl)
    Y_ar = H.alloc(pa, s.TENSOR_C)
    pa.run(H_r, W2_r, Y_ar, H.workspace(pa))
    for y in Y_ar:
        s.shmm_layernorm(y, gam, bet, y, eps=1e-5)
    s.shmm_sync_status()
    torch.cuda.synchronize()
    for a, b in zip(Y_n, Y_ar):
        assert torch.equal(a, b)
    # oracle chain
    Xn, W1n, W2n = X.float().numpy(), W1.float().numpy(), W2.float().numpy()
    _, hres = oracle.sharded_matmul(X8, ((), ()), ((), ("X",)), ((), ("X",)), Xn, W1n, "bf16", gelu=True,
                                    nthreads=8)
    Hn = np.zeros((T, F), np.float32)
    for r, ((i0, k0), blk) in hres.items():
        Hn[i0:i0 + blk.shape[0], k0:k0 + blk.shape[1]] = blk
    _, yres = oracle.sharded_matmul(X8, ((), ("X",)), (("X",), ()), (("X",), ()), Hn, W2n, "bf16", nthreads=8)
    Yn = np.zeros((T, D), np.float32)
    for r, ((i0, k0), blk) in yres.items():
        Yn[i0:i0 + blk.shape[0]] = blk
    ref = oracle.layernorm(Yn, gam.cpu().numpy(), bet.cpu().numpy(), 1e-5, "bf16")
    for y in Y_n:
        got = y.float().cpu().numpy()
        assert np.abs(got - ref).max() <= BF16_TOL * np.abs(ref).max()


@pytest.mark.parametrize("pair", KERNELS)
@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("mesh,sA,sB,sC,I,J,K", [
    (Y2, ((), ("Y",)), (("Y",), ()), (("Y",), ()), 300, 2000, 264),          # J_r = 1000 = 15 k-blocks + 40
    (XY42, (("X",), ("Y",)), (("Y",), ()), (("X",), ()), 1040, 1808, 520),  # J_r = 904, M_r = 260
])
def test_ragged_contraction(s, pair, fused, mesh, sA, sB, sC, I, J, K, monkeypatch):
    """Per-rank contraction lengths that are not a multiple of the 64-wide
    k-block (the last block is zero-filled by TMA), with ragged M and N, on
    both GEMM kernels, fused and unfused, against the oracle."""
    use_kernel(monkeypatch, pair)
    A, B = shmm_inputs.scaled_normal_pair(I, J, K, "bf16", seed=I + K)
    plan, gpu = run_gpu(mesh, sA, sB, sC, A, B, "bf16", "f32", s.FLAG_FUSED if fused else 0)
    assert plan.info.tensor_core == 1
    _, ores = oracle_run(mesh, sA, sB, sC, A, B, "f32")
    compare(plan, gpu, ores, exact=False, tol=F32P_TOL)


@pytest.mark.parametrize("case,sA,sB,sC", FOUR)
@pytest.mark.parametrize("limit", [2, 34, 150])
def test_sm_limit_keeps_the_bits(s, case, sA, sB, sC, limit, monkeypatch):
    """A plan capped to a few SMs (one CTA pair, a share of the GPU, odd and
    above the pair count) gives the same bits as the plan on every SM, in
    both tile widths, while other plans run on their own streams beside it."""
    from partial_sum_reduction_gb300 import helpers as H
    A, B = shmm_inputs.scaled_normal_pair(1024, 512, 768, "bf16", seed=case + 40)
    for wide in ("0", "1"):
        monkeypatch.setenv("SHMM_TC_WIDE", wide)
        outs = []
        for lim in (0, limit):
            plan = s.Plan(XY22, sA, sB, sC, 1024, 512, 768, "bf16", "bf16", s.FLAG_FUSED)
            plan.set_sm_limit(lim)
            A_r, B_r = H.shard(plan, s.TENSOR_A, A), H.shard(plan, s.TENSOR_B, B)
            C_r = H.alloc(plan, s.TENSOR_C, fill=float("nan"))
            side = torch.cuda.Stream()
            other = s.Plan(XY22, sA, sB, sC, 1024, 512, 768, "bf16", "bf16", s.FLAG_FUSED)
            other.set_sm_limit(max(2, 152 - limit))
            oC = H.alloc(other, s.TENSOR_C)
            side.wait_stream(torch.cuda.current_stream())
            other.run(A_r, B_r, oC, H.workspace(other), stream=side)
            plan.run(A_r, B_r, C_r, H.workspace(plan))
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            outs.append([c.cpu() for c in C_r])
            for c, o in zip(C_r, oC):
                assert torch.equal(c, o)
        for a, b in zip(*outs):
            assert torch.equal(a, b)


@pytest.mark.parametrize("pair", ["pair_wide", "single"])
def test_gelu_epilogue_against_the_tanh_form(s, pair, monkeypatch):
    """The epilogue's GeLU, x s(2u) (the tanh form through the logistic
    identity: one hardware exponential, the reciprocal by Newton-Raphson on
    the FMA pipe), against torch's tanh-form GeLU
    evaluated in fp32 on the same pre-activations: the GEMM's own fp32
    output without GeLU.  Pre-activations span about +-12, so both tails
    and the zero crossing are hit."""
    from partial_sum_reduction_gb300 import helpers as H
    use_kernel(monkeypatch, pair)
    I, J, K = 512, 256, 8 * 512
    A = shmm_inputs.normal_matrix((I, J), 1.0, "bf16", seed=60)
    B = shmm_inputs.normal_matrix((J, K), 4.0 / J ** 0.5, "bf16", seed=61)
    outs = []
    for fl in (0, s.FLAG_GELU):
        p = s.Plan(X8, ((), ()), ((), ("X",)), ((), ("X",)), I, J, K, "bf16", "f32", fl)
        A_r, B_r = H.shard(p, s.TENSOR_A, A), H.shard(p, s.TENSOR_B, B)
        C_r = H.alloc(p, s.TENSOR_C, fill=float("nan"))
        p.run(A_r, B_r, C_r, H.workspace(p))
        torch.cuda.synchronize()
        outs.append(C_r)
    span = max(float(c.abs().max()) for c in outs[0])
    assert span > 8.0
    for pre, got in zip(*outs):
        ref = torch.nn.functional.gelu(pre, approximate="tanh")
        assert torch.all((got - ref).abs() <= 1e-5 * ref.abs() + 1e-6), float((got - ref).abs().max())


@pytest.mark.parametrize("wide", ["0", "1", None])
def test_run_batch_equals_separate_runs(s, wide, monkeypatch):
    """Independent plans through shmm_run_batch give the bits of their own
    shmm_run calls: the four cases (in-place gathers, a fused reduce-scatter)
    sharing one launch, a GeLU plan with fp32 output, a rank-order fused
    all-reduce, a plan whose local M fits one 128-row tile (single-CTA
    kernel), and an unfused reduction that runs through shmm_run; more
    operand slots than one launch holds, so the joined plans take two."""
    from partial_sum_reduction_gb300 import helpers as H
    if wide is None:
        monkeypatch.delenv("SHMM_TC_WIDE", raising=False)
    else:
        monkeypatch.setenv("SHMM_TC_WIDE", wide)
    A, B = shmm_inputs.scaled_normal_pair(1024, 512, 768, "bf16", seed=50)
    specs = [(XY22, sA, sB, sC, "bf16", s.FLAG_FUSED, A, B) for _, sA, sB, sC in FOUR]
    A2, B2 = shmm_inputs.scaled_normal_pair(512, 256, 1024, "bf16", seed=51)
    specs.append((X8, ((), ()), ((), ("X",)), ((), ("X",)), "f32", s.FLAG_GELU, A2, B2))
    A3, B3 = shmm_inputs.scaled_normal_pair(1024, 1024, 512, "bf16", seed=52)
    specs.append((XY42, (("X",), ("Y",)), (("Y",), ()), (("X",), ()), "bf16", s.FLAG_FUSED | s.FLAG_RANK_ORDER,
                  A3, B3))
    A4, B4 = shmm_inputs.scaled_normal_pair(256, 512, 320, "bf16", seed=53)
    specs.append((XY22, (("X",), ()), ((), ("Y",)), (("X",), ("Y",)), "bf16", 0, A4, B4))   # local M = 128
    specs.append((XY22, ((), ("Y",)), (("Y",), ()), (("Y",), ()), "bf16", 0, A, B))       # unfused reduction
    plans, ins, refs, outs, wss = [], [], [], [], []
    for mesh, sA, sB, sC, odt, fl, a, b in specs:
        I, J = a.shape
        K = b.shape[1]
        p = s.Plan(mesh, sA, sB, sC, I, J, K, "bf16", odt, fl)
        A_r, B_r = H.shard(p, s.TENSOR_A, a), H.shard(p, s.TENSOR_B, b)
        ref = H.alloc(p, s.TENSOR_C, fill=float("nan"))
        p.run(A_r, B_r, ref, H.workspace(p))
        plans.append(p)
        ins.append((A_r, B_r))
        refs.append(ref)
        outs.append(H.alloc(p, s.TENSOR_C, fill=float("nan")))
        wss.append(H.workspace(p))
    launches = s.shmm_kernel_launches()
    s.shmm_run_batch(plans, [x[0] for x in ins], [x[1] for x in ins], outs, wss)
    s.shmm_sync_status()
    torch.cuda.synchronize()
    launched = s.shmm_kernel_launches() - launches
    # eight plans, seven of them joined: no more kernels than one per plan
    assert launched < len(plans)
    for i, (o, r) in enumerate(zip(outs, refs)):
        for q, (x, y) in enumerate(zip(o, r)):
            assert not torch.isnan(x.float()).any(), "plan %d rank %d unwritten" % (i, q)
            assert torch.equal(x, y), "plan %d rank %d differs from its own shmm_run" % (i, q)


def test_run_batch_more_plans_than_one_launch_holds(s):
    """Six joined plans: more segments than one launch carries, so the batch
    takes two launches; the same plan appears twice with different outputs;
    every plan carries an SM limit, so each launch takes the largest.  Each
    output equals the plan's own shmm_run bit for bit."""
    from partial_sum_reduction_gb300 import helpers as H
    plans, ins, refs, outs = [], [], [], []
    shapes = [(512, 256, 320), (768, 512, 256), (512, 128, 512), (1024, 256, 264), (512, 256, 320)]
    for i, (I, J, K) in enumerate(shapes):
        A, B = shmm_inputs.scaled_normal_pair(I, J, K, "bf16", seed=70 + i)
        p = s.Plan(Y2, ((), ("Y",)), (("Y",), ()), ((), ()), I, J, K, "bf16", "bf16", s.FLAG_FUSED)
        p.set_sm_limit(40 + 8 * i)
        A_r, B_r = H.shard(p, s.TENSOR_A, A), H.shard(p, s.TENSOR_B, B)
        ref = H.alloc(p, s.TENSOR_C, fill=float("nan"))
        p.run(A_r, B_r, ref)
        copies = 2 if i == 0 else 1   # plan 0 twice, each time into its own outputs
        for _ in range(copies):
            plans.append(p)
            ins.append((A_r, B_r))
            refs.append(ref)
            outs.append(H.alloc(p, s.TENSOR_C, fill=float("nan")))
    launches = s.shmm_kernel_launches()
    s.shmm_run_batch(plans, [x[0] for x in ins], [x[1] for x in ins], outs)
    s.shmm_sync_status()
    torch.cuda.synchronize()
    assert s.shmm_kernel_launches() - launches == 2
    for i, (o, r) in enumerate(zip(outs, refs)):
        for x, y in zip(o, r):
            assert torch.equal(x, y), "plan %d" % i


@pytest.mark.parametrize("flags", ["FUSED", "FUSED|RANK_ORDER", "0"])
def test_repeated_runs_give_identical_bits(s, flags):
    """Every path is deterministic: one input gives one result, run after run
    (fixed reduction orders, no atomics), through shmm_run and shmm_run_host."""
    from partial_sum_reduction_gb300 import helpers as H
    fl = 0
    for f in flags.split("|"):
        fl |= getattr(s, "FLAG_" + f) if f != "0" else 0
    I, J, K = 1024, 2048, 768
    A, B = shmm_inputs.scaled_normal_pair(I, J, K, "bf16", seed=31)
    p = s.Plan(XY42, (("X",), ("Y",)), (("Y",), ()), (("X",), ()), I, J, K, "bf16", "bf16", fl)
    A_r, B_r, ws = H.shard(p, s.TENSOR_A, A), H.shard(p, s.TENSOR_B, B), H.workspace(p)
    first = None
    for _ in range(5):
        C_r = H.alloc(p, s.TENSOR_C, fill=float("nan"))
        p.run(A_r, B_r, C_r, ws)
        torch.cuda.synchronize()
        bits = torch.cat([c.flatten() for c in C_r]).view(torch.int16).cpu()
        first = bits if first is None else first
        assert torch.equal(bits, first)
    C_h = torch.empty(I, K, dtype=torch.bfloat16).pin_memory()
    C_r = H.alloc(p, s.TENSOR_C, fill=float("nan"))
    p.run_host(A.pin_memory(), B.pin_memory(), C_h, H.alloc(p, s.TENSOR_A), H.alloc(p, s.TENSOR_B), C_r, ws)
    s.shmm_sync_status()
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([c.flatten() for c in C_r]).view(torch.int16).cpu(), first)
