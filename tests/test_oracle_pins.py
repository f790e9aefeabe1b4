"""Pins the CPU oracle to facts outside itself: values the pages print
(tests/golden/), closed forms, IEEE-754 facts, library routines and brute
force.  No GPU."""
import itertools

import numpy as np
import pytest
import torch

import oracle
import shmm_inputs
from conftest import load_golden

Y2 = [("Y", 2)]
XY22 = [("X", 2), ("Y", 2)]
XY42 = [("X", 4), ("Y", 2)]


def _parse_mesh(s):
    return [(a.split(":")[0].strip(), int(a.split(":")[1])) for a in s.split(",")]


def _parse_spec(s):
    """'I_X,J_Y' -> (('X',), ('Y',)); 'I_XY' -> (('X','Y'),); 'K' -> ()."""
    dims = []
    for d in s.split(","):
        d = d.strip()
        dims.append(tuple(d.split("_", 1)[1]) if "_" in d else ())
    return tuple(dims)


def _stitch(mesh, plan, result, I, K):
    """Rebuilds the global C from every rank's owned box; checks that all
    ranks that hold an element agree bitwise."""
    C = np.full((I, K), np.nan)
    for r, ((i0, k0), blk) in result.items():
        sub = C[i0:i0 + blk.shape[0], k0:k0 + blk.shape[1]]
        seen = ~np.isnan(sub)
        assert np.array_equal(sub[seen], blk[seen]), "replicas disagree"
        C[i0:i0 + blk.shape[0], k0:k0 + blk.shape[1]] = blk
    assert not np.isnan(C).any(), "some element of C is owned by no rank"
    return C


# ----------------------------------------------------------- worked example

def test_worked_example_partials_and_collectives():
    g = load_golden("p2_worked_example.txt")
    mesh = _parse_mesh(g["mesh"])
    A = np.array(g["A"], np.float32)
    B = np.array(g["B"], np.float32)
    sA, sB = ((), ("Y",)), (("Y",), ())
    _, parts = oracle.partials(mesh, sA, sB, A, B)
    assert parts[0][1].tolist() == g["partial_rank0"]
    assert parts[1][1].tolist() == g["partial_rank1"]
    plan, rs = oracle.sharded_matmul(mesh, sA, sB, (("Y",), ()), A, B)
    assert plan.case == 3 and plan.collective == "reduce_scatter"
    assert rs[0][1].tolist() == g["reduce_scatter_rank0"] and rs[0][0] == (0, 0)
    assert rs[1][1].tolist() == g["reduce_scatter_rank1"] and rs[1][0] == (1, 0)
    # all-gather of the finished rows: every rank holds the whole C
    gathered = oracle.all_gather([rs[0][1], rs[1][1]], dim=0)
    for blk in gathered:
        assert blk.tolist() == g["all_gather_every_rank"]
    plan, ar = oracle.sharded_matmul(mesh, sA, sB, ((), ()), A, B)
    assert plan.collective == "all_reduce"
    for r in (0, 1):
        assert ar[r][1].tolist() == g["all_gather_every_rank"]


def test_worked_example_payload_bytes():
    g = load_golden("p2_worked_example.txt")
    mesh = _parse_mesh(g["mesh"])
    sA, sB = ((), ("Y",)), (("Y",), ())
    rs = oracle.payload_bytes(mesh, sA, sB, (("Y",), ()), 2, 2, 2, "f32", "f32")
    assert rs["reduce_scatter"] == g["reduce_scatter_payload_bytes_per_rank"]
    ar = oracle.payload_bytes(mesh, sA, sB, ((), ()), 2, 2, 2, "f32", "f32")
    assert ar["result_all_gather"] == g["all_gather_payload_bytes_per_rank"]
    assert ar["per_rank"] == g["payload_bytes_per_rank"]
    assert ar["total"] == g["payload_bytes_total"]


# Operand all-gather payload, counted by hand at the sender ("Sharded matrix
# multiplication and result ownership", Engineering example: a sent payload
# counts once; "Sharding Matrix Multiply", AllGather: every member ends with
# the whole operand, so each rank sends its own shard to the G-1 others).
# I = J = K = 2048, bf16 (2 bytes).
OPERAND_AG_BY_HAND = [
    # case 2 on {X:2,Y:2}: A[I,J_X] -> shard [2048,1024] = 4 MiB, one peer
    (XY22, ((), ("X",)), ((), ()), ((), ()), 2048 * 1024 * 2 * 1),
    # case 4 on {X:2,Y:2}: B[J,K_X] -> shard [2048,1024] = 4 MiB, one peer
    (XY22, (("X",), ()), ((), ("X",)), (("X",), ()), 2048 * 1024 * 2 * 1),
    # case 2 on {X:4,Y:2}: A[I,J_X] -> shard [2048,512] = 2 MiB, three peers
    (XY42, ((), ("X",)), ((), ()), ((), ()), 2048 * 512 * 2 * 3),
    # case 2, both operands J-sharded on different axes: A[I,J_X] shard
    # [2048,1024] to one X peer, B[J_Y,K] shard [1024,2048] to one Y peer
    (XY22, ((), ("X",)), (("Y",), ()), ((), ()), 2048 * 1024 * 2 + 1024 * 2048 * 2),
    # case 3 with case 4's gather: B[J_Y,K_X] shard [1024,1024] = 2 MiB,
    # gathered over X along K to one peer; A[I_X,J_Y] is not moved
    (XY22, (("X",), ("Y",)), (("Y",), ("X",)), (("X",), ()), 1024 * 1024 * 2 * 1),
]


@pytest.mark.parametrize("mesh,sA,sB,sC,expected", OPERAND_AG_BY_HAND)
def test_operand_all_gather_payload_by_hand(mesh, sA, sB, sC, expected):
    pay = oracle.payload_bytes(mesh, sA, sB, sC, 2048, 2048, 2048, "bf16", "bf16")
    assert pay["operand_all_gather"] == expected


@pytest.mark.parametrize("mesh,sA,sB,sC,expected", OPERAND_AG_BY_HAND)
def test_operand_all_gather_payload_counted_at_the_receivers(mesh, sA, sB, sC, expected):
    """The same bytes counted the other way, on small shapes: every element a
    rank holds after the gather but not before was received from a peer, and
    every byte received was sent once, so the total over ranks must equal N
    times the per-rank sent payload."""
    I, J, K = 8, 16, 24
    N = oracle.mesh_size(mesh)
    plan = oracle.plan_matmul(mesh, sA, sB, sC)
    received = 0
    for before, after, shape in ((sA, plan.local_A, (I, J)), (sB, plan.local_B, (J, K))):
        for r in range(N):
            (b0, b1), (bn0, bn1) = oracle.shard_box(mesh, before, shape, r)
            (a0, a1), (an0, an1) = oracle.shard_box(mesh, after, shape, r)
            for i in range(a0, a0 + an0):
                for j in range(a1, a1 + an1):
                    if not (b0 <= i < b0 + bn0 and b1 <= j < b1 + bn1):
                        received += 2
    pay = oracle.payload_bytes(mesh, sA, sB, sC, I, J, K, "bf16", "bf16")
    assert pay["operand_all_gather"] * N == received
    assert received > 0


def test_concatenating_partials_is_not_the_result():
    g = load_golden("p2_worked_example.txt")
    cat = np.concatenate([np.array(g["partial_rank0"]), np.array(g["partial_rank1"])])
    assert cat.shape[0] == g["concatenated_partials_rows"]
    C = np.array(g["all_gather_every_rank"])
    assert not np.array_equal(cat[:2], C) and not np.array_equal(cat[2:], C)


# --------------------------------------------------- identity and brute force

CASES = [
    # (mesh, A spec, B spec, C spec, expected case, expected collective)
    (Y2, ((), ("Y",)), (("Y",), ()), (("Y",), ()), 3, "reduce_scatter"),
    (Y2, ((), ("Y",)), (("Y",), ()), ((), ("Y",)), 3, "reduce_scatter"),
    (Y2, ((), ("Y",)), (("Y",), ()), ((), ()), 3, "all_reduce"),
    (XY22, (("X",), ()), ((), ("Y",)), (("X",), ("Y",)), 1, "none"),
    (XY22, (("X",), ()), ((), ("Y",)), ((), ()), 1, "none"),
    (XY22, ((), ("X",)), ((), ()), ((), ()), 2, "none"),
    (XY22, ((), ("Y",)), (("Y",), ()), (("Y",), ()), 3, "reduce_scatter"),
    (XY22, (("X",), ()), ((), ("X",)), (("X",), ()), 4, "none"),
    (XY42, (("X",), ("Y",)), (("Y",), ()), (("X",), ()), 3, "all_reduce"),
    (XY42, (("X",), ("Y",)), (("Y",), ()), (("X", "Y"), ()), 3, "reduce_scatter"),
    (XY42, (("X",), ("Y",)), (("Y",), ()), ((), ()), 3, "all_reduce"),
    (XY22, ((), ("X", "Y")), (("X", "Y"), ()), ((), ()), 3, "all_reduce"),
    (XY22, ((), ("X", "Y")), (("X", "Y"), ()), (("X", "Y"), ()), 3, "reduce_scatter"),
]


@pytest.mark.parametrize("mesh,sA,sB,sC,case,coll", CASES)
def test_sum_of_partials_equals_dense_product(mesh, sA, sB, sC, case, coll):
    """Row Parallelism: Y = sum_i X_i A_i, and every ownership assembles the
    dense product; exact on small integers."""
    I, J, K = 16, 24, 8
    A, B = shmm_inputs.split_k_integer(I, J, K, seed=3)
    A, B = A.numpy(), B.numpy()
    plan, res = oracle.sharded_matmul(mesh, sA, sB, sC, A, B)
    assert plan.case == case and plan.collective == coll
    C = _stitch(mesh, plan, res, I, K)
    assert np.array_equal(C, A.astype(np.float64) @ B.astype(np.float64))
    # and sum over one reduction group of the raw partials is the product
    _, parts = oracle.partials(mesh, sA, sB, A, B)
    grp = oracle.reduction_group(mesh, plan, 0)
    (i0, k0), P0 = parts[0]
    tot = sum(parts[q][1].astype(np.float64) for q in grp)
    ref = A.astype(np.float64) @ B.astype(np.float64)
    assert np.array_equal(tot, ref[i0:i0 + P0.shape[0], k0:k0 + P0.shape[1]])


def test_brute_force_tiny_shapes():
    """Every tiny shape and split against the library matmul."""
    rng = np.random.default_rng(7)
    for n in (1, 2, 4):
        mesh = [("Y", n)]
        for I, Jb, K in itertools.product(range(1, 4), range(1, 3), range(1, 4)):
            J = Jb * n
            A = rng.integers(-3, 4, (I, J)).astype(np.float32)
            B = rng.integers(-3, 4, (J, K)).astype(np.float32)
            for sC in (((), ()),) + ((((("Y",), ()),) if I % n == 0 else ())):
                plan, res = oracle.sharded_matmul(mesh, ((), ("Y",)), (("Y",), ()), sC, A, B)
                C = _stitch(mesh, plan, res, I, K)
                assert np.array_equal(C, A.astype(np.float64) @ B.astype(np.float64))


def test_local_product_matches_library_on_floats():
    rng = np.random.default_rng(11)
    A = rng.standard_normal((37, 53)).astype(np.float32)
    B = rng.standard_normal((53, 29)).astype(np.float32)
    P = oracle.local_product(A, B)
    ref = (A.astype(np.float64) @ B.astype(np.float64)).astype(np.float32)
    np.testing.assert_allclose(P, ref, rtol=2e-7, atol=1e-6)
    # row sampling returns exactly the rows of the full product
    rows = [0, 5, 36, 17]
    np.testing.assert_array_equal(oracle.local_product(A, B, rows=rows), P[rows])
    # threading does not change any element
    np.testing.assert_array_equal(oracle.local_product(A, B, nthreads=4), P)
    assert np.array_equal(oracle.dense_product_f64(A, B), A.astype(np.float64) @ B.astype(np.float64))


def test_sampled_rows_match_full_result():
    A, B = shmm_inputs.scaled_normal_pair(32, 16, 24, dtype="bf16", seed=5)
    A, B = A.float().numpy(), B.float().numpy()
    for sC in ((("X", "Y"), ()), (("X",), ())):
        plan, full = oracle.sharded_matmul(XY42, (("X",), ("Y",)), (("Y",), ()), sC, A, B,
                                           out_dtype="bf16")
        rows = [0, 3, 9, 31, 16]
        _, samp = oracle.sharded_matmul(XY42, (("X",), ("Y",)), (("Y",), ()), sC, A, B,
                                        out_dtype="bf16", rows=rows)
        for r, (crow, k0, blk) in samp.items():
            (i0, fk0), fblk = full[r]
            assert k0 == fk0
            np.testing.assert_array_equal(blk, fblk[crow - i0])


# ---------------------------------------------------------- planner facts

def test_down_projection_shapes_and_bytes():
    g = load_golden("p4_down_projection.txt")
    mesh = _parse_mesh(g["mesh"])
    sA, sB = _parse_spec(g["A_spec"]), _parse_spec(g["B_spec"])
    I = g["A_blocks"][0] * g["A_shard"][0]
    J = g["A_blocks"][1] * g["A_shard"][1]
    K = g["B_block"][1] * g["B_blocks"][1]
    assert oracle.mesh_size(mesh) == g["devices"]
    _, ext = oracle.shard_box(mesh, sA, (I, J), 0)
    assert list(ext) == g["A_shard"]
    assert round(oracle.shard_bytes(mesh, sA, (I, J), "bf16") / 1e6, 1) == g["A_bytes_per_device_MB"]
    boxes = [oracle.shard_box(mesh, sA, (I, J), r) for r in range(8)]
    assert max(boxes.count(b) for b in boxes) == g["A_copies_of_each_shard"]
    assert len(set(boxes)) == g["A_blocks"][0] * g["A_blocks"][1]
    bboxes = {oracle.shard_box(mesh, sB, (J, K), r) for r in range(8)}
    assert len(bboxes) == g["B_blocks"][0] * g["B_blocks"][1]
    assert all(list(b[1]) == g["B_block"] for b in bboxes)
    plan = oracle.plan_matmul(mesh, sA, sB, (("X",), ()))
    assert plan.case == g["case"] and plan.collective == "all_reduce" and plan.unreduced == ("Y",)
    assert round(oracle.shard_bytes(mesh, plan.out_C, (I, K), "bf16") / 1e6, 1) == g["C_bytes_per_device_MB"]
    assert round(oracle.local_flops(mesh, sA, sB, I, J, K) / 1e9) == g["local_matmul_GFLOP"]
    rep = _parse_spec(g["replicated_A_spec"])
    rboxes = [oracle.shard_box(mesh, rep, (I, J), r) for r in range(8)]
    assert min(rboxes.count(b) for b in rboxes) == g["replicated_A_copies"]


def test_rank_numbering_first_axis_major():
    assert oracle.rank_coords(XY42, 5) == {"X": 2, "Y": 1}
    assert oracle.rank_of(XY42, {"X": 3, "Y": 0}) == 6
    # I_XY: X major -> rank (x, y) holds block 2x + y
    for r in range(8):
        c = oracle.rank_coords(XY42, r)
        (i0, _), (n, _) = oracle.shard_box(XY42, (("X", "Y"), ()), (64, 4), r)
        assert i0 == (2 * c["X"] + c["Y"]) * 8 and n == 8
        (i0, _), _ = oracle.shard_box(XY42, (("Y", "X"), ()), (64, 4), r)
        assert i0 == (4 * c["Y"] + c["X"]) * 8


def test_validity_rules():
    with pytest.raises(ValueError):
        oracle.plan_matmul(XY22, (("X",), ("X",)), ((), ()), ((), ()))   # A[I_X, J_X]
    with pytest.raises(ValueError):
        oracle.plan_matmul(XY22, (("X",), ()), ((), ("X",)), (("X",), ("X",)))  # C[I_X, K_X]
    with pytest.raises(ValueError):
        oracle.plan_matmul(XY22, (("Z",), ()), ((), ()), ((), ()))
    with pytest.raises(ValueError):
        oracle.shard_box(XY22, (("X",), ()), (3, 4), 0)  # uneven split


def test_four_cases_of_the_cheat_sheet():
    assert oracle.plan_matmul(XY22, (("X",), ()), ((), ("Y",)), (("X",), ("Y",))).case == 1
    p2 = oracle.plan_matmul(XY22, ((), ("X",)), ((), ()), ((), ()))
    assert p2.case == 2 and p2.gather_A == ("X",) and p2.unreduced == ()
    p3 = oracle.plan_matmul(XY22, ((), ("Y",)), (("Y",), ()), ((), ()))
    assert p3.case == 3 and p3.unreduced == ("Y",)
    p4 = oracle.plan_matmul(XY22, (("X",), ()), ((), ("X",)), (("X",), ()))
    assert p4.case == 4 and p4.gather_B == ("X",) and p4.local_B == ((), ())
    # without the gather, rank x could only form the diagonal block C[x, x]
    for r in range(4):
        (ai, _), _ = oracle.shard_box(XY22, (("X",), ()), (8, 8), r)
        (_, bk), _ = oracle.shard_box(XY22, ((), ("X",)), (8, 8), r)
        assert ai == bk


# ------------------------------------------------------ rounding and order

def test_bf16_rounding_against_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    specials = np.array([0.0, -0.0, 1.0, np.inf, -np.inf, 3.3895314e38, 1e-40, -1e-45,
                         1.00390625, 1.01171875, 1.0000001], np.float32)
    x = np.concatenate([x, specials])
    ours = oracle.round_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(ours.view(np.uint32), ref.view(np.uint32))
    # ties go to the even neighbour (closed form)
    assert oracle.round_bf16(np.float32(1.00390625))[()] == 1.0          # 1 + 2^-8
    assert oracle.round_bf16(np.float32(1.01171875))[()] == 1.015625     # 1 + 3*2^-8
    assert np.isnan(oracle.round_bf16(np.float32(np.nan))[()])


def test_summation_order_is_the_declared_one():
    """fp32 facts: 2^24 + 1 rounds back to 2^24, 2^24 + 2 is exact."""
    parts = [np.array([2.0 ** 24], np.float32)] + [np.array([1.0], np.float32)] * 3
    assert oracle.sum_partials(parts, "sequential")[0] == 2.0 ** 24
    assert oracle.sum_partials(parts, "pairwise")[0] == 2.0 ** 24 + 2
    parts = [np.array([-0.0], np.float32)] * 3
    s = oracle.sum_partials(parts, "pairwise")
    assert s[0] == 0.0 and np.signbit(s[0])   # -0 padding keeps -0


def test_all_reduce_is_reduce_scatter_then_all_gather():
    bufs = [b.numpy().reshape(8, 16) for b in shmm_inputs.partial_buffers(4, 128, "f32", seed=2)]
    ar = oracle.collective_reduce(bufs, "all_reduce", "bf16")
    rs = oracle.collective_reduce(bufs, "reduce_scatter", "bf16", scatter_dim=0)
    ag = oracle.all_gather(rs, dim=0)
    for a, b in zip(ar, ag):
        np.testing.assert_array_equal(a, b)
    rs1 = oracle.collective_reduce(bufs, "reduce_scatter", "f32", scatter_dim=1)
    ag1 = oracle.all_gather(rs1, dim=1)
    np.testing.assert_array_equal(ag1[0], oracle.collective_reduce(bufs, "all_reduce", "f32")[0])


def test_gelu_closed_forms_and_library():
    x = np.linspace(-8, 8, 4001).astype(np.float32)
    gp, gm = oracle.gelu_tanh(x).astype(np.float64), oracle.gelu_tanh(-x).astype(np.float64)
    assert oracle.lib().orc_gelu_tanh(0.0) == 0.0
    # tanh is odd, so gelu(x) - gelu(-x) = x
    np.testing.assert_allclose(gp - gm, x, rtol=0, atol=2e-6)
    assert abs(oracle.lib().orc_gelu_tanh(20.0) - 20.0) < 1e-12
    assert abs(oracle.lib().orc_gelu_tanh(-20.0)) < 1e-12
    ref = torch.nn.functional.gelu(torch.from_numpy(x).double(), approximate="tanh").numpy()
    # agree with the library to rounding: the two evaluate 1 + tanh(.) with
    # different libm tanh calls, which differ by an ulp where it cancels
    np.testing.assert_allclose(oracle.gelu_tanh(x), ref.astype(np.float32), rtol=2e-7, atol=1e-12)


# ------------------------------------------- planted mistakes get caught

def _runs_pins():
    test_worked_example_partials_and_collectives()
    for args in CASES:
        test_sum_of_partials_equals_dense_product(*args)
    test_down_projection_shapes_and_bytes()
    test_rank_numbering_first_axis_major()
    test_summation_order_is_the_declared_one()


@pytest.mark.parametrize("mutation", ["drop_last_rank", "transpose_B", "minor_axis_major",
                                      "skip_all_reduce_copies", "double_sum"])
def test_planted_mistakes_fail_a_pin(monkeypatch, mutation):
    if mutation == "drop_last_rank":
        orig = oracle.sum_partials
        monkeypatch.setattr(oracle, "sum_partials",
                            lambda parts, order="sequential": orig(parts[:-1] or parts, order))
    elif mutation == "transpose_B":
        orig = oracle.local_product
        # B's buffer read as if it were stored K-major (a transposed operand)
        monkeypatch.setattr(oracle, "local_product",
                            lambda A, B, **kw: orig(A, np.ascontiguousarray(
                                np.asarray(B).reshape(np.asarray(B).shape[::-1]).T), **kw))
    elif mutation == "minor_axis_major":
        def coords(mesh, r):
            c = {}
            for name, size in mesh:
                c[name] = r % size
                r //= size
            return c
        monkeypatch.setattr(oracle, "rank_coords", coords)
    elif mutation == "skip_all_reduce_copies":
        orig = oracle.plan_matmul

        def plan(*a):
            p = orig(*a)
            if p.collective == "all_reduce":
                p.collective = "reduce_scatter"
            return p
        monkeypatch.setattr(oracle, "plan_matmul", plan)
    elif mutation == "double_sum":
        orig = oracle.sum_partials
        monkeypatch.setattr(oracle, "sum_partials",
                            lambda parts, order="sequential": orig(list(parts) + [parts[0]], order))
    with pytest.raises(AssertionError):
        _runs_pins()


def test_all_to_all_moves_which_dim_is_sharded():
    """A[I,J_X] -> A[I_X,J] on two ranks, by hand: rank 0 holds column 0
    and ends with row 0; rank 1 holds column 1 and ends with row 1."""
    mesh = [("X", 2)]
    src = {0: np.array([[0.0], [2.0]]), 1: np.array([[1.0], [3.0]])}
    out = oracle.reshard(mesh, ((), ("X",)), (("X",), ()), src, (2, 2))
    assert out[0].tolist() == [[0.0, 1.0]] and out[1].tolist() == [[2.0, 3.0]]
    # dropping the axis is the all-gather
    full = oracle.reshard(mesh, ((), ("X",)), ((), ()), src, (2, 2))
    assert full[0].tolist() == full[1].tolist() == [[0.0, 1.0], [2.0, 3.0]]
    # replicas of one block (ranks 0 and 1 on {X:2,Y:2}) must agree
    with pytest.raises(ValueError):
        oracle.reshard([("X", 2), ("Y", 2)], ((), ("X",)), ((), ()),
                       {0: np.zeros((2, 1)), 1: np.ones((2, 1)), 2: np.ones((2, 1)), 3: np.ones((2, 1))},
                       (2, 2))


def test_layernorm_closed_form_invariants_and_library():
    x = np.array([[1.0, 2.0, 3.0, 4.0]], np.float32)
    y = oracle.layernorm(x, np.ones(4), np.zeros(4), eps=0.0)
    np.testing.assert_allclose(y[0], np.array([-1.5, -0.5, 0.5, 1.5]) / np.sqrt(1.25), rtol=1e-6)
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((16, 300)) * 3 + 1).astype(np.float32)
    y = oracle.layernorm(x, np.ones(300), np.zeros(300), eps=1e-5).astype(np.float64)
    np.testing.assert_allclose(y.mean(axis=1), 0, atol=1e-6)
    np.testing.assert_allclose(y.var(axis=1), 1, atol=1e-5)
    g = rng.standard_normal(300).astype(np.float32)
    b = rng.standard_normal(300).astype(np.float32)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x).double(), (300,), torch.from_numpy(g).double(),
                                         torch.from_numpy(b).double(), eps=1e-5).numpy()
    np.testing.assert_allclose(oracle.layernorm(x, g, b, 1e-5), ref.astype(np.float32), rtol=1e-6, atol=1e-6)
    # shifting or scaling a row leaves its normalised form unchanged
    np.testing.assert_allclose(oracle.layernorm(5 * x + 7, g, b, 0.0), oracle.layernorm(x, g, b, 0.0),
                               rtol=0, atol=2e-5)
