"""CPU oracle for the sharded matmul A[I,J] . B[J,K] -> C[I,K] and its
partial-sum reduction -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA path
(``partial_sum_reduction_gb300``) and neither imports the other; the only
module both sides use is ``shmm_inputs`` (seeded input generation, none of
the method's arithmetic).

The oracle is the plain definition of the method, step by step as
"Sharded matrix multiplication and result ownership" (The mechanism, steps
1-6) lays it out:

1. declare the complete shapes, the mesh and each tensor's sharding;
2. give each rank its shard of A and of B (after an AllGather of the operand
   where the case needs one: "Sharding Matrix Multiply", Case 2 and Case 4);
3. form each rank's local product over its slice of the contracted dim with
   a triple loop (``oracle.c``: double accumulation, fp32 partial);
4. add the partials with matching output coordinates over each reduction
   group, in ascending rank order in fp32, rounded once to the output dtype;
5. hand each rank the block its ownership names: reduce-scatter keeps the
   owner's block, all-reduce every member's full copy, all-gather the
   concatenation of owner blocks.

Notation follows "Sharded matmuls and collectives on a torus" (Notation):
a mesh is a list of (axis name, size) pairs, rank id is row-major over the
axes with the first axis major; a sharding gives, per array dim, the tuple
of mesh axes that split it (several axes flatten with the first listed
major, as in I_XY).

Where the pages leave a step open, the oracle reads it plainly: a
reduce-scatter splits the dim the requested C sharding extends (rows in the
worked example); a replicated operand is one buffer per rank; every rank
computes its own product; partials are fp32 and are added in ascending rank
order; GeLU is the tanh form; uneven shards are rejected.  Every function
below is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import itertools
import math
import os
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

from . import build as _build

_LIB = None


def lib():
    """Loads liboracle.so, compiling it first when it is missing or stale."""
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        L.orc_round_bf16.argtypes = [ctypes.c_float]
        L.orc_round_bf16.restype = ctypes.c_float
        L.orc_round_bf16_array.argtypes = [f32p, f32p, i64]
        L.orc_local_product.argtypes = [f32p, i64, f32p, i64, f32p, i64, i64,
                                        ctypes.POINTER(ctypes.c_int64), i64, i64, ctypes.c_int]
        L.orc_dense_product_f64.argtypes = [f64p, f64p, f64p, i64, i64, i64]
        L.orc_sum_sequential.argtypes = [ctypes.POINTER(f32p), ctypes.c_int, i64, f32p]
        L.orc_sum_pairwise.argtypes = [ctypes.POINTER(f32p), ctypes.c_int, i64, f32p]
        L.orc_gelu_tanh.argtypes = [ctypes.c_double]
        L.orc_gelu_tanh.restype = ctypes.c_double
        L.orc_gelu_tanh_array.argtypes = [f32p, f32p, i64]
        _LIB = L
    return _LIB


def _fp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _f32c(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


# ---------------------------------------------------------------- arithmetic

def round_bf16(x) -> np.ndarray:
    """fp32 -> nearest bfloat16 (ties to even), returned as fp32 values."""
    a = _f32c(x)
    out = np.empty_like(a)
    lib().orc_round_bf16_array(_fp(a), _fp(out), a.size)
    return out


def gelu_tanh(x) -> np.ndarray:
    """GeLU, tanh form, evaluated in double and stored as fp32
    ("The simple maths behind parallel training", MLP block)."""
    a = _f32c(x)
    out = np.empty_like(a)
    lib().orc_gelu_tanh_array(_fp(a), _fp(out), a.size)
    return out


def local_product(A, B, rows: Optional[Sequence[int]] = None, nthreads: int = 1) -> np.ndarray:
    """One rank's local product P = A . B over its slice of the contracted
    dim (the partial C_r of "Sharded matrix multiplication and result
    ownership", step 3; Z_i = X_i A_i in "Row Parallelism").  Triple loop,
    double accumulation in ascending j, fp32 result.  ``rows`` restricts the
    output to the listed rows of A (sampled outputs)."""
    A = _f32c(A)
    B = _f32c(B)
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("local_product: shapes %s . %s do not contract" % (A.shape, B.shape))
    J, K = B.shape
    if rows is None:
        nrows, rp = A.shape[0], None
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        if r.size and (r.min() < 0 or r.max() >= A.shape[0]):
            raise ValueError("local_product: row index out of range")
        nrows, rp = r.size, r.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    P = np.empty((nrows, K), dtype=np.float32)
    if nrows and K:
        lib().orc_local_product(_fp(A), A.shape[1], _fp(B), K, _fp(P), K, nrows, rp, J, K,
                                int(nthreads))
    return P


def dense_product_f64(A, B) -> np.ndarray:
    """Unrounded dense product in double (checks "sum of partials = A.B")."""
    A = np.ascontiguousarray(np.asarray(A, dtype=np.float64))
    B = np.ascontiguousarray(np.asarray(B, dtype=np.float64))
    I, J = A.shape
    K = B.shape[1]
    D = np.empty((I, K), dtype=np.float64)
    dp = ctypes.POINTER(ctypes.c_double)
    lib().orc_dense_product_f64(A.ctypes.data_as(dp), B.ctypes.data_as(dp), D.ctypes.data_as(dp),
                                I, J, K)
    return D


def sum_partials(parts: Sequence[np.ndarray], order: str = "sequential") -> np.ndarray:
    """Sum of partials with matching coordinates.  ``sequential``: fp32,
    ascending rank, ((p0+p1)+p2)+... (the canonical order); ``pairwise``:
    balanced binary tree over the ranks in ascending order."""
    ps = [_f32c(p) for p in parts]
    if not ps:
        raise ValueError("sum_partials: no partials")
    shape = ps[0].shape
    for p in ps:
        if p.shape != shape:
            raise ValueError("sum_partials: partial shapes differ")
    out = np.empty(shape, dtype=np.float32)
    arr = (ctypes.POINTER(ctypes.c_float) * len(ps))(*[_fp(p) for p in ps])
    fn = {"sequential": lib().orc_sum_sequential, "pairwise": lib().orc_sum_pairwise}[order]
    fn(arr, len(ps), out.size, _fp(out))
    return out


def to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """Rounds fp32 values to the stored element type ("f32" or "bf16")."""
    if dtype == "f32":
        return _f32c(x)
    if dtype == "bf16":
        return round_bf16(x)
    raise ValueError("unknown dtype %r" % dtype)


ELEM_BYTES = {"f32": 4, "bf16": 2}

# ----------------------------------------------------------- mesh and specs

Mesh = List[Tuple[str, int]]
Spec = Tuple[Tuple[str, ...], Tuple[str, ...]]


def mesh_size(mesh: Mesh) -> int:
    return int(np.prod([s for _, s in mesh])) if mesh else 1


def rank_coords(mesh: Mesh, r: int) -> Dict[str, int]:
    """Coordinates of rank r: row-major over the axes, first axis major."""
    coords = {}
    for name, size in reversed(mesh):
        coords[name] = r % size
        r //= size
    return coords


def rank_of(mesh: Mesh, coords: Dict[str, int]) -> int:
    r = 0
    for name, size in mesh:
        r = r * size + coords[name]
    return r


def check_spec(mesh: Mesh, spec: Spec, what: str) -> None:
    """A mesh axis may split at most one dim of an array; A[I_X, J_X] is
    invalid ("Sharding Matrix Multiply", Notation, Rule)."""
    names = {n for n, _ in mesh}
    seen = set()
    for axes in spec:
        for a in axes:
            if a not in names:
                raise ValueError("%s: unknown mesh axis %r" % (what, a))
            if a in seen:
                raise ValueError("%s: mesh axis %r shards more than one dim" % (what, a))
            seen.add(a)


def shard_box(mesh: Mesh, spec: Spec, shape: Tuple[int, int], r: int):
    """(offsets, extents) of rank r's block of a 2-D array under ``spec``.
    A dim split by axes (a1, a2, ...) has prod(sizes) contiguous blocks; the
    block index flattens the rank's coordinates with a1 major.  Axes not
    named replicate the array.  Uneven splits are rejected."""
    sizes = dict(mesh)
    c = rank_coords(mesh, r)
    off, ext = [], []
    for d, axes in enumerate(spec):
        n = 1
        idx = 0
        for a in axes:
            n *= sizes[a]
            idx = idx * sizes[a] + c[a]
        if shape[d] % n:
            raise ValueError("dim %d of size %d does not split %d ways" % (d, shape[d], n))
        blk = shape[d] // n
        off.append(idx * blk)
        ext.append(blk)
    return tuple(off), tuple(ext)


def _is_prefix(p: Tuple[str, ...], q: Tuple[str, ...]) -> bool:
    return tuple(q[:len(p)]) == tuple(p)


@dataclass
class MatmulPlan:
    """The oracle's own reading of a sharded matmul (independent of the
    C++ planner)."""
    case: int
    local_A: Spec          # A's sharding after any operand all-gather
    local_B: Spec
    gather_A: Tuple[str, ...]   # axes A is all-gathered over (case 2/4)
    gather_B: Tuple[str, ...]
    natural_C: Spec        # sharding of the local product, before reduction
    unreduced: Tuple[str, ...]  # {U_...}: axes the partials still sum over
    collective: str        # "none", "reduce_scatter" or "all_reduce"
    scatter_dim: int       # dim the reduce-scatter splits (-1 if none)
    reduced_C: Spec        # ownership after the reduction (owner blocks)
    out_C: Spec            # ownership the consumer asked for
    gather_C: Tuple[str, ...] = field(default_factory=tuple)  # result all-gather axes


def plan_matmul(mesh: Mesh, sA: Spec, sB: Spec, sC: Spec) -> MatmulPlan:
    """Classifies A[I,J].B[J,K] into the four cases ("Sharding Matrix
    Multiply", Case 1-4 and Summary; "Sharded matmuls and collectives on a
    torus", The four cases) and derives the collective the requested output
    ownership needs ("Sharded matrix multiplication and result ownership",
    step 4: all-reduce for a replicated C, reduce-scatter for disjoint
    shards; step 5: all-gather only when the consumer needs the whole)."""
    check_spec(mesh, sA, "A")
    check_spec(mesh, sB, "B")
    check_spec(mesh, sC, "C")
    (aI, aJ), (bJ, bK) = sA, sB
    gather_A: Tuple[str, ...] = ()
    gather_B: Tuple[str, ...] = ()
    if aJ and aJ == bJ:
        case = 3
        U = tuple(aJ)
    elif aJ or bJ:
        case = 2                      # AllGather the J-sharded operand(s)
        gather_A, gather_B = tuple(aJ), tuple(bJ)
        aJ, bJ, U = (), (), ()
    else:
        case = 1
        U = ()
    if set(aI) & set(bK):
        # a shared mesh axis on both non-contracting dims would give only the
        # diagonal blocks; AllGather B along K first (Case 4)
        if case == 1:
            case = 4
        gather_B = tuple(gather_B) + tuple(bK)
        bK = ()
    natural = (tuple(aI), tuple(bK))
    cI, cK = tuple(sC[0]), tuple(sC[1])
    if U:
        inI = [a for a in U if a in cI]
        inK = [a for a in U if a in cK]
        if inI and inK:
            raise ValueError("C: the reduced axes may scatter over one dim only")
        if inI or inK:
            d = 0 if inI else 1
            reduced = list(natural)
            reduced[d] = natural[d] + U
            reduced = (reduced[0], reduced[1])
            collective, scatter_dim = "reduce_scatter", d
        else:
            reduced, collective, scatter_dim = natural, "all_reduce", -1
    else:
        reduced, collective, scatter_dim = natural, "none", -1
    if not (_is_prefix(cI, reduced[0]) and _is_prefix(cK, reduced[1])):
        raise ValueError("C: requested ownership %r is not reachable from %r by reduction and "
                         "all-gather" % (sC, reduced))
    gather_C = tuple(reduced[0][len(cI):]) + tuple(reduced[1][len(cK):])
    return MatmulPlan(case=case, local_A=(tuple(aI), tuple(aJ)), local_B=(tuple(bJ), tuple(bK)),
                      gather_A=gather_A, gather_B=gather_B, natural_C=natural, unreduced=U,
                      collective=collective, scatter_dim=scatter_dim, reduced_C=reduced,
                      out_C=(cI, cK), gather_C=gather_C)


def _group(mesh: Mesh, r: int, free_axes: Sequence[str]) -> List[int]:
    """Ranks that agree with r on every axis outside ``free_axes``, ascending."""
    c = rank_coords(mesh, r)
    sizes = dict(mesh)
    ranks = []
    for vals in itertools.product(*[range(sizes[a]) for a in free_axes]):
        cc = dict(c)
        cc.update(zip(free_axes, vals))
        ranks.append(rank_of(mesh, cc))
    return sorted(ranks)


def reduction_group(mesh: Mesh, plan: MatmulPlan, r: int) -> List[int]:
    """Ranks whose partials add into rank r's result: those differing from
    r only on the unreduced (contracted) axes."""
    return _group(mesh, r, plan.unreduced)


def sharded_matmul(mesh: Mesh, sA: Spec, sB: Spec, sC: Spec, A, B, out_dtype: str = "f32",
                   gelu: bool = False, order: str = "sequential",
                   rows: Optional[Sequence[int]] = None, nthreads: int = 1):
    """Runs the method on global arrays A [I,J] and B [J,K] (fp32 values,
    already rounded to the input dtype) and returns, per rank, the block of C
    it owns: ``{rank: (offsets, array)}``.

    ``rows``: restrict to these global rows of C (sampled outputs); the
    returned arrays then hold only those rows that fall in each rank's box,
    as ``{rank: (row_indices, col_offset, array)}``.
    ``gelu``: apply GeLU to the finished sum before the output rounding (the
    column-parallel first matmul of the MLP pair).
    """
    A = _f32c(A)
    B = _f32c(B)
    I, J = A.shape
    J2, K = B.shape
    if J != J2:
        raise ValueError("A and B do not contract")
    plan = plan_matmul(mesh, sA, sB, sC)
    N = mesh_size(mesh)
    row_set = None if rows is None else np.asarray(sorted(set(int(x) for x in rows)), np.int64)

    # steps 2-3: each rank's operands (after any all-gather) and local product
    partial = {}
    for r in range(N):
        (ai0, aj0), (ain, ajn) = shard_box(mesh, plan.local_A, (I, J), r)
        (bj0, bk0), (bjn, bkn) = shard_box(mesh, plan.local_B, (J, K), r)
        if (aj0, ajn) != (bj0, bjn):
            raise AssertionError("A and B slices of J differ on rank %d" % r)
        Ar = A[ai0:ai0 + ain, aj0:aj0 + ajn]
        Br = B[bj0:bj0 + bjn, bk0:bk0 + bkn]
        if row_set is None:
            local_rows = None
            grows = np.arange(ai0, ai0 + ain)
        else:
            grows = row_set[(row_set >= ai0) & (row_set < ai0 + ain)]
            local_rows = grows - ai0
        partial[r] = (grows, bk0, local_product(Ar, Br, rows=local_rows, nthreads=nthreads))

    # step 4: sum over each reduction group (ascending rank), owner blocks
    owned = {}
    for r in range(N):
        group = reduction_group(mesh, plan, r)
        grows, k0, _ = partial[r]
        S = sum_partials([partial[q][2] for q in group], order=order)
        if gelu:
            S = gelu_tanh(S)
        S = to_dtype(S, out_dtype)
        (o_i0, o_k0), (o_in, o_kn) = shard_box(mesh, plan.reduced_C, (I, K), r)
        sel = (grows >= o_i0) & (grows < o_i0 + o_in)
        owned[r] = (grows[sel], o_k0, S[sel][:, o_k0 - k0:o_k0 - k0 + o_kn])

    # step 5: deliver the requested ownership (all-gather of owner blocks)
    result = {}
    for r in range(N):
        (c_i0, c_k0), (c_in, c_kn) = shard_box(mesh, plan.out_C, (I, K), r)
        if row_set is None:
            crow = np.arange(c_i0, c_i0 + c_in)
        else:
            crow = row_set[(row_set >= c_i0) & (row_set < c_i0 + c_in)]
        out = np.full((crow.size, c_kn), np.nan, dtype=np.float32)
        for q in _group(mesh, r, plan.gather_C):
            qrows, q_k0, blk = owned[q]
            for li, g in enumerate(qrows):
                pos = np.searchsorted(crow, g)
                if pos < crow.size and crow[pos] == g:
                    out[pos, q_k0 - c_k0:q_k0 - c_k0 + blk.shape[1]] = blk[li]
        if row_set is None:
            result[r] = ((c_i0, c_k0), out)
        else:
            result[r] = (crow, c_k0, out)
    return plan, result


def partials(mesh: Mesh, sA: Spec, sB: Spec, A, B, nthreads: int = 1):
    """Each rank's unreduced local product P_r (fp32) with its box offset:
    ``{rank: ((i0, k0), P_r)}`` -- the C[...]{U} state before the reduction."""
    A = _f32c(A)
    B = _f32c(B)
    I, J = A.shape
    K = B.shape[1]
    # the local operands do not depend on C's ownership: plan against a
    # replicated C request, which every case accepts
    probe = plan_matmul(mesh, sA, sB, ((), ()))
    out = {}
    for r in range(mesh_size(mesh)):
        (ai0, aj0), (ain, ajn) = shard_box(mesh, probe.local_A, (I, J), r)
        (bj0, bk0), (bjn, bkn) = shard_box(mesh, probe.local_B, (J, K), r)
        out[r] = ((ai0, bk0), local_product(A[ai0:ai0 + ain, aj0:aj0 + ajn],
                                            B[bj0:bj0 + bjn, bk0:bk0 + bkn], nthreads=nthreads))
    return probe, out


def collective_reduce(parts: Sequence[np.ndarray], mode: str, dtype: str, order: str = "sequential",
                      scatter_dim: int = 0):
    """The collective alone, on one reduction group's partial buffers (all of
    one shape): ``reduce_scatter`` returns the owner blocks (owner q gets
    block q of ``scatter_dim``), ``all_reduce`` every member's full copy
    ("Sharding Matrix Multiply", Communication primitives)."""
    S = to_dtype(sum_partials(parts, order=order), dtype)
    G = len(parts)
    if mode == "all_reduce":
        return [S.copy() for _ in range(G)]
    if mode == "reduce_scatter":
        n = S.shape[scatter_dim]
        if n % G:
            raise ValueError("reduce_scatter: dim does not split evenly")
        b = n // G
        if scatter_dim == 0:
            return [S[q * b:(q + 1) * b].copy() for q in range(G)]
        return [S[:, q * b:(q + 1) * b].copy() for q in range(G)]
    raise ValueError(mode)


def all_gather(shards: Sequence[np.ndarray], dim: int = 0):
    """Every member gets the concatenation of the shards in rank order
    ("Sharding Matrix Multiply", AllGather)."""
    full = np.concatenate([_f32c(s) for s in shards], axis=dim)
    return [full.copy() for _ in shards]


def payload_bytes(mesh: Mesh, sA: Spec, sB: Spec, sC: Spec, I: int, J: int, K: int,
                  in_dtype: str, out_dtype: str, partial_dtype: str = "f32") -> Dict[str, int]:
    """Bytes each rank SENDS, counted once at the sender ("Sharded matrix
    multiplication and result ownership", step 6 and the Engineering
    example): a collective over a group of G ranks on an array of V bytes
    per rank makes each rank send the (G-1) blocks of V/G it does not keep
    (reduce-scatter) or its own block to the G-1 others (all-gather)."""
    plan = plan_matmul(mesh, sA, sB, sC)
    sizes = dict(mesh)

    def gsize(axes):
        return int(np.prod([sizes[a] for a in axes])) if axes else 1

    out = {"operand_all_gather": 0, "reduce_scatter": 0, "result_all_gather": 0}
    eb_in = ELEM_BYTES[in_dtype]
    for axes, spec, shape in ((plan.gather_A, plan.local_A, (I, J)),
                              (plan.gather_B, plan.local_B, (J, K))):
        if axes:
            _, ext = shard_box(mesh, spec, shape, 0)
            G = gsize(axes)
            out["operand_all_gather"] += (G - 1) * (ext[0] * ext[1] // G) * eb_in
    _, pext = shard_box(mesh, plan.natural_C, (I, K), 0)
    V = pext[0] * pext[1]
    if plan.unreduced:
        G = gsize(plan.unreduced)
        out["reduce_scatter"] = (G - 1) * (V // G) * ELEM_BYTES[partial_dtype]
        if plan.collective == "all_reduce":
            # all-reduce = reduce-scatter + all-gather of the finished blocks
            out["result_all_gather"] += (G - 1) * (V // G) * ELEM_BYTES[out_dtype]
    if plan.gather_C:
        _, rext = shard_box(mesh, plan.reduced_C, (I, K), 0)
        G = gsize(plan.gather_C)
        out["result_all_gather"] += (G - 1) * rext[0] * rext[1] * ELEM_BYTES[out_dtype]
    out["per_rank"] = sum(out.values())
    out["total"] = out["per_rank"] * mesh_size(mesh)
    return out


def shard_bytes(mesh: Mesh, spec: Spec, shape, dtype: str) -> int:
    _, ext = shard_box(mesh, spec, shape, 0)
    return ext[0] * ext[1] * ELEM_BYTES[dtype]


def local_flops(mesh: Mesh, sA: Spec, sB: Spec, I: int, J: int, K: int) -> int:
    """2 * I_r * J_r * K_r, the multiply-adds of one rank's local product."""
    plan = plan_matmul(mesh, sA, sB, ((), ()))
    (_, _), (ain, ajn) = shard_box(mesh, plan.local_A, (I, J), 0)
    (_, _), (_, bkn) = shard_box(mesh, plan.local_B, (J, K), 0)
    return 2 * ain * ajn * bkn


def reshard(mesh: Mesh, spec_from: Spec, spec_to: Spec, shards_from: Dict[int, np.ndarray],
            shape: Tuple[int, int]) -> Dict[int, np.ndarray]:
    """AllToAll / reshard ("Sharding Matrix Multiply", Communication
    primitives: move which dim is sharded, A[I,J_X] -> A[I_X,J]): rebuild
    the array from every rank's block under ``spec_from`` (replicas must
    agree), then hand each rank its block under ``spec_to``."""
    check_spec(mesh, spec_from, "from")
    check_spec(mesh, spec_to, "to")
    full = np.full(shape, np.nan, dtype=np.float64)
    for r, blk in shards_from.items():
        (i0, j0), (n0, n1) = shard_box(mesh, spec_from, shape, r)
        blk = np.asarray(blk, dtype=np.float64)
        if blk.shape != (n0, n1):
            raise ValueError("rank %d: block shape %s, expected %s" % (r, blk.shape, (n0, n1)))
        sub = full[i0:i0 + n0, j0:j0 + n1]
        seen = ~np.isnan(sub)
        if not np.array_equal(sub[seen], blk[seen]):
            raise ValueError("replicated source blocks disagree")
        full[i0:i0 + n0, j0:j0 + n1] = blk
    if np.isnan(full).any():
        raise ValueError("source blocks do not cover the array")
    out = {}
    for r in range(mesh_size(mesh)):
        (i0, j0), (n0, n1) = shard_box(mesh, spec_to, shape, r)
        out[r] = full[i0:i0 + n0, j0:j0 + n1].copy()
    return out


def layernorm(x, gamma, beta, eps: float = 1e-5, out_dtype: str = "f32") -> np.ndarray:
    """Layer normalisation of every row (a token) over its features, as the
    sequence-parallel block applies it locally per token ("The simple maths
    behind parallel training", Sequence parallelism); the form of Ba, Kiros &
    Hinton (2016): y = (x - mean) / sqrt(var + eps) * gamma + beta with the
    mean and the biased variance of the row, evaluated in double and rounded
    once to ``out_dtype``."""
    x = np.asarray(x, dtype=np.float64)
    g = np.asarray(gamma, dtype=np.float64)
    b = np.asarray(beta, dtype=np.float64)
    mean = x.mean(axis=1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=1, keepdims=True)
    y = (x - mean) / np.sqrt(var + eps) * g + b
    return to_dtype(y.astype(np.float32), out_dtype)
