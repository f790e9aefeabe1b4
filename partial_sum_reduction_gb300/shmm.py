"""ctypes binding of libshmm (include/shmm.h): the same entry points, with
argument marshalling only.  Every step of the sharded matmul runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback, and importing a
missing library raises.

Meshes and shardings may be given as Python values or as strings:
  mesh   [("X", 4), ("Y", 2)]  or  "{X:4,Y:2}"
  spec   (("X",), ("Y",))  or  "P('X','Y')"  or  "P(('X','Y'),None)"  or
         the subscript form "I_X,J_Y" ("Sharded matmuls and collectives on a
         torus", Notation: A[I_X, J_Y] is P('X', 'Y'); A[I_XY, J] is
         P(('X', 'Y'), None)).
Tensors are lists of per-rank CUDA tensors, indexed by rank id, each a dense
row-major buffer holding exactly that rank's box (Plan.rank_box).
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import List, Optional, Sequence, Tuple

HERE = os.path.dirname(os.path.abspath(__file__))
# SHMM_CHECKED=1 selects the bounds-checked build (build.build(checked=True)):
# the same kernels with every global index compared with its buffer's extent.
LIB_PATH = os.path.join(HERE, "libshmm_checked.so" if os.environ.get("SHMM_CHECKED") == "1" else "libshmm.so")

MAX_AXES = 8
MAX_RANKS = 256

# status codes
OK, ERR_INVALID_SPEC, ERR_ILLEGAL_OUTPUT, ERR_SHAPE, ERR_DTYPE, ERR_NULL, ERR_ALIGN, ERR_CUDA, \
    ERR_TIMEOUT, ERR_NOMEM, ERR_UNSUPPORTED, ERR_INJECTED, ERR_BOUNDS = range(13)
F32, BF16 = 0, 1
FLAG_FUSED, FLAG_GELU, FLAG_TREE, FLAG_PARTIAL_OUT_DTYPE, FLAG_SIMT = 0x1, 0x2, 0x4, 0x8, 0x10
FLAG_RANK_ORDER = 0x20
TENSOR_A, TENSOR_B, TENSOR_C, TENSOR_P, TENSOR_A_LOCAL, TENSOR_B_LOCAL, TENSOR_C_REDUCED = range(7)
COLL_NONE, COLL_REDUCE_SCATTER, COLL_ALL_REDUCE = range(3)
COLLECTIVE_NAMES = {COLL_NONE: "none", COLL_REDUCE_SCATTER: "reduce_scatter",
                    COLL_ALL_REDUCE: "all_reduce"}
DTYPE_CODES = {"f32": F32, "bf16": BF16}


class shmm_mesh_t(ctypes.Structure):
    _fields_ = [("naxes", ctypes.c_int), ("name", (ctypes.c_char * 8) * MAX_AXES),
                ("size", ctypes.c_int * MAX_AXES)]


class shmm_spec_t(ctypes.Structure):
    _fields_ = [("naxes", ctypes.c_int * 2), ("axes", (ctypes.c_int * MAX_AXES) * 2)]


class shmm_plan_info_t(ctypes.Structure):
    _fields_ = [("case_id", ctypes.c_int), ("collective", ctypes.c_int),
                ("scatter_dim", ctypes.c_int), ("nranks", ctypes.c_int),
                ("group_size", ctypes.c_int), ("ngroups", ctypes.c_int),
                ("gather_A_size", ctypes.c_int), ("gather_B_size", ctypes.c_int),
                ("gather_C_size", ctypes.c_int), ("in_dtype", ctypes.c_int),
                ("out_dtype", ctypes.c_int), ("partial_dtype", ctypes.c_int),
                ("flags", ctypes.c_uint32), ("tensor_core", ctypes.c_int), ("fused", ctypes.c_int),
                ("local_I", ctypes.c_int64), ("local_J", ctypes.c_int64), ("local_K", ctypes.c_int64),
                ("flops_per_rank", ctypes.c_int64), ("payload_operand_ag", ctypes.c_int64),
                ("payload_reduce_scatter", ctypes.c_int64), ("payload_result_ag", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_size_t), ("fused_gather", ctypes.c_int)]


class shmm_device_model_t(ctypes.Structure):
    _fields_ = [("flops_per_s", ctypes.c_double), ("bytes_per_s", ctypes.c_double)]


class shmm_operand_choice_t(ctypes.Structure):
    _fields_ = [("choice", ctypes.c_int), ("gather_compute_bound", ctypes.c_int),
                ("bytes_gather", ctypes.c_double), ("bytes_reduce", ctypes.c_double),
                ("t_gather", ctypes.c_double), ("t_reduce", ctypes.c_double)]


class ShmmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (_status_name(status), message))
        self.status = status


EXPORTS = ["shmm_plan", "shmm_plan_destroy", "shmm_plan_query", "shmm_plan_rank_box",
           "shmm_plan_set_sm_limit", "shmm_plan_group", "shmm_workspace_size", "shmm_local_matmul", "shmm_reduce_scatter",
           "shmm_all_reduce", "shmm_all_gather", "shmm_run", "shmm_sync_status", "shmm_last_error",
           "shmm_status_string", "shmm_version", "shmm_kernel_launches", "shmm_run_static_workspace",
           "shmm_selftest_wait_timeout", "shmm_choose_operand", "shmm_reshard", "shmm_layernorm",
           "shmm_layernorm_all_gather", "shmm_run_host", "shmm_bounds_checked", "shmm_run_batch"]

_lib = None


def lib():
    """The loaded libshmm.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("%s is not built (%s); run partial_sum_reduction_gb300.build.build(%s)"
                               % (os.path.basename(LIB_PATH), LIB_PATH,
                                  "checked=True" if LIB_PATH.endswith("_checked.so") else ""))
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        PP = ctypes.POINTER(ctypes.c_void_p)
        st = ctypes.c_int
        L.shmm_plan.argtypes = [ctypes.POINTER(shmm_mesh_t), ctypes.POINTER(shmm_spec_t),
                                ctypes.POINTER(shmm_spec_t), ctypes.POINTER(shmm_spec_t),
                                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                ctypes.c_int, ctypes.c_uint32, ctypes.POINTER(P)]
        L.shmm_plan_destroy.argtypes = [P]
        L.shmm_plan_set_sm_limit.argtypes = [P, ctypes.c_int]
        L.shmm_plan_query.argtypes = [P, ctypes.POINTER(shmm_plan_info_t)]
        L.shmm_plan_rank_box.argtypes = [P, ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]
        L.shmm_plan_group.argtypes = [P, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
        L.shmm_workspace_size.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
        L.shmm_local_matmul.argtypes = [P, PP, PP, PP, P]
        L.shmm_reduce_scatter.argtypes = [P, PP, PP, P]
        L.shmm_all_reduce.argtypes = [P, PP, PP, P]
        L.shmm_all_gather.argtypes = [P, ctypes.c_int, PP, PP, P]
        L.shmm_run.argtypes = [P, PP, PP, PP, P, ctypes.c_size_t, P]
        L.shmm_run_static_workspace.argtypes = [P, PP, PP, PP, P]
        L.shmm_run_batch.argtypes = [ctypes.c_int, PP, ctypes.POINTER(PP), ctypes.POINTER(PP), ctypes.POINTER(PP),
                                     PP, ctypes.POINTER(ctypes.c_size_t), P]
        L.shmm_run_host.argtypes = [P, P, P, P, PP, PP, PP, P, ctypes.c_size_t, P]
        L.shmm_sync_status.argtypes = [P]
        L.shmm_selftest_wait_timeout.argtypes = [ctypes.c_uint64, P]
        L.shmm_layernorm.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int, P, P, P, ctypes.c_float, P, P]
        L.shmm_layernorm_all_gather.argtypes = [P, PP, P, P, ctypes.c_float, PP, P]
        L.shmm_reshard.argtypes = [ctypes.POINTER(shmm_mesh_t), ctypes.POINTER(shmm_spec_t),
                                   ctypes.POINTER(shmm_spec_t), ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                   PP, PP, P]
        L.shmm_choose_operand.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                          ctypes.c_int, ctypes.POINTER(shmm_device_model_t),
                                          ctypes.POINTER(shmm_operand_choice_t)]
        L.shmm_last_error.restype = ctypes.c_char_p
        L.shmm_status_string.argtypes = [ctypes.c_int]
        L.shmm_status_string.restype = ctypes.c_char_p
        L.shmm_kernel_launches.restype = ctypes.c_uint64
        for f in EXPORTS:
            if f not in ("shmm_last_error", "shmm_status_string", "shmm_kernel_launches"):
                getattr(L, f).restype = st
        _lib = L
    return _lib


def _status_name(s: int) -> str:
    try:
        return lib().shmm_status_string(s).decode()
    except Exception:  # library unavailable while formatting an error
        return "status %d" % s


def _check(status: int) -> None:
    if status != OK:
        raise ShmmError(status, lib().shmm_last_error().decode())


# ------------------------------------------------------------- parsing (D6)

def parse_mesh(mesh) -> List[Tuple[str, int]]:
    """'{X:4,Y:2}' or [('X',4),('Y',2)] -> [('X',4),('Y',2)]."""
    if isinstance(mesh, str):
        body = mesh.strip().strip("{}")
        out = []
        for part in body.split(","):
            if part.strip():
                name, size = part.split(":")
                out.append((name.strip().strip("'\""), int(size)))
        return out
    return [(str(n), int(s)) for n, s in mesh]


def parse_spec(spec) -> Tuple[Tuple[str, ...], Tuple[str, ...]]:
    """Sharding of a 2-D array in any of the accepted forms -> per-dim axis
    tuples, first axis major."""
    if isinstance(spec, str):
        s = spec.strip()
        if s.startswith("P(") and s.endswith(")"):
            inner = s[2:-1].strip()
            if not inner:
                return ((), ())
            dims = []
            depth, cur = 0, ""
            for ch in inner + ",":
                if ch == "," and depth == 0:
                    dims.append(cur.strip())
                    cur = ""
                    continue
                depth += ch == "("
                depth -= ch == ")"
                cur += ch
            parsed = []
            for d in dims:
                if d in ("None", ""):
                    parsed.append(())
                else:
                    parsed.append(tuple(re.findall(r"['\"]([^'\"]+)['\"]", d)))
            while len(parsed) < 2:
                parsed.append(())
            if len(parsed) != 2:
                raise ValueError("a 2-D PartitionSpec has at most two entries: %r" % spec)
            return parsed[0], parsed[1]
        dims = [d.strip() for d in s.strip("[]").split(",")]
        if len(dims) != 2:
            raise ValueError("expected two dims in %r" % spec)
        return tuple(tuple(d.split("_", 1)[1]) if "_" in d else () for d in dims)
    a, b = spec
    return tuple(a), tuple(b)


def _mesh_struct(mesh) -> shmm_mesh_t:
    m = shmm_mesh_t()
    axes = parse_mesh(mesh)
    if len(axes) > MAX_AXES:
        raise ValueError("at most %d mesh axes" % MAX_AXES)
    m.naxes = len(axes)
    for i, (n, s) in enumerate(axes):
        enc = n.encode()
        if len(enc) >= 8:
            raise ValueError("axis name %r longer than 7 bytes" % n)
        m.name[i].value = enc
        m.size[i] = s
    return m


def _spec_struct(mesh, spec) -> shmm_spec_t:
    names = [n for n, _ in parse_mesh(mesh)]
    s = shmm_spec_t()
    for d, axes in enumerate(parse_spec(spec)):
        if len(axes) > MAX_AXES:
            raise ValueError("too many axes on one dim")
        s.naxes[d] = len(axes)
        for i, a in enumerate(axes):
            s.axes[d][i] = names.index(a) if a in names else 99  # 99: rejected by the planner
    return s


# --------------------------------------------------------------- marshalling

def _ptr_array(tensors: Sequence, what: str) -> ctypes.Array:
    arr = (ctypes.c_void_p * len(tensors))()
    for i, t in enumerate(tensors):
        if t is None:
            arr[i] = None
        elif isinstance(t, int):
            arr[i] = t
        else:
            arr[i] = t.data_ptr()
    return arr


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """A shmm_plan_t handle (freed on garbage collection or close())."""

    def __init__(self, mesh, spec_A, spec_B, spec_C, I: int, J: int, K: int, in_dtype: str = "bf16",
                 out_dtype: str = "bf16", flags: int = 0):
        self.mesh = parse_mesh(mesh)
        self.spec_A, self.spec_B, self.spec_C = parse_spec(spec_A), parse_spec(spec_B), parse_spec(spec_C)
        self.shape = (int(I), int(J), int(K))
        self.in_dtype, self.out_dtype, self.flags = in_dtype, out_dtype, int(flags)
        h = ctypes.c_void_p()
        m = _mesh_struct(self.mesh)
        sa, sb, sc = (_spec_struct(self.mesh, s) for s in (self.spec_A, self.spec_B, self.spec_C))
        _check(lib().shmm_plan(ctypes.byref(m), ctypes.byref(sa), ctypes.byref(sb), ctypes.byref(sc),
                               int(I), int(J), int(K), DTYPE_CODES[in_dtype], DTYPE_CODES[out_dtype],
                               int(flags), ctypes.byref(h)))
        self._h = h
        self.info = self.query()
        self.nranks = self.info.nranks

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            lib().shmm_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def set_sm_limit(self, max_sms: int):
        """Caps the SMs this plan's tensor-core GEMM launches occupy (0: all)."""
        _check(lib().shmm_plan_set_sm_limit(self._h, int(max_sms)))

    def query(self) -> shmm_plan_info_t:
        info = shmm_plan_info_t()
        _check(lib().shmm_plan_query(self._h, ctypes.byref(info)))
        return info

    def rank_box(self, tensor: int, rank: int):
        off = (ctypes.c_int64 * 2)()
        ext = (ctypes.c_int64 * 2)()
        _check(lib().shmm_plan_rank_box(self._h, tensor, rank, off, ext))
        return (off[0], off[1]), (ext[0], ext[1])

    def group(self, rank: int) -> List[int]:
        out = (ctypes.c_int * self.info.group_size)()
        _check(lib().shmm_plan_group(self._h, rank, out))
        return list(out)

    def workspace_size(self) -> int:
        n = ctypes.c_size_t()
        _check(lib().shmm_workspace_size(self._h, ctypes.byref(n)))
        return n.value

    # ---- device work ----
    def local_matmul(self, A_r, B_r, P_r, stream=None):
        _check(lib().shmm_local_matmul(self._h, _ptr_array(A_r, "A"), _ptr_array(B_r, "B"),
                                       _ptr_array(P_r, "P"), _stream_handle(stream)))

    def reduce_scatter(self, P_r, C_r, stream=None):
        _check(lib().shmm_reduce_scatter(self._h, _ptr_array(P_r, "P"), _ptr_array(C_r, "C"),
                                         _stream_handle(stream)))

    def all_reduce(self, P_r, C_r, stream=None):
        _check(lib().shmm_all_reduce(self._h, _ptr_array(P_r, "P"), _ptr_array(C_r, "C"),
                                     _stream_handle(stream)))

    def all_gather(self, tensor: int, shard_r, full_r, stream=None):
        _check(lib().shmm_all_gather(self._h, tensor, _ptr_array(shard_r, "shard"),
                                     _ptr_array(full_r, "full"), _stream_handle(stream)))

    def run(self, A_r, B_r, C_r, workspace=None, stream=None):
        ws_ptr = None if workspace is None else (workspace if isinstance(workspace, int) else workspace.data_ptr())
        ws_bytes = 0 if workspace is None else (
            self.workspace_size() if isinstance(workspace, int) else workspace.numel() * workspace.element_size())
        _check(lib().shmm_run(self._h, _ptr_array(A_r, "A"), _ptr_array(B_r, "B"), _ptr_array(C_r, "C"),
                              ws_ptr, ws_bytes, _stream_handle(stream)))

    def layernorm_all_gather(self, shard_r, gamma, beta, full_r, eps: float = 1e-5, stream=None):
        """Layer-normalise the row-owned result blocks and all-gather them
        (sequence parallelism's LayerNorm then AllGather, in one pass)."""
        _check(lib().shmm_layernorm_all_gather(self._h, _ptr_array(shard_r, "shard"), gamma.data_ptr(),
                                               beta.data_ptr(), float(eps), _ptr_array(full_r, "full"),
                                               _stream_handle(stream)))

    def run_host(self, A_host, B_host, C_host, A_r, B_r, C_r, workspace=None, stream=None):
        """shmm_run_host: global A [I,J], B [J,K] (CPU tensors, pinned for
        overlap, or None when A_r / B_r already hold the shards) in, global C
        [I,K] (a CPU tensor, or None) out, through the ranks' device buffers."""
        def host_ptr(t, shape, what):
            if t is None:
                return None
            if (not hasattr(t, "data_ptr") or t.device.type != "cpu" or not t.is_contiguous()
                    or tuple(t.shape) != shape):
                raise ValueError("%s_host must be a contiguous CPU tensor of shape %s" % (what, shape))
            return t.data_ptr()
        ws_ptr = None if workspace is None else (workspace if isinstance(workspace, int) else workspace.data_ptr())
        ws_bytes = 0 if workspace is None else (
            self.workspace_size() if isinstance(workspace, int) else workspace.numel() * workspace.element_size())
        I, J, K = self.shape
        _check(lib().shmm_run_host(self._h, host_ptr(A_host, (I, J), "A"), host_ptr(B_host, (J, K), "B"),
                                   host_ptr(C_host, (I, K), "C"),
                                   _ptr_array(A_r, "A"), _ptr_array(B_r, "B"), _ptr_array(C_r, "C"),
                                   ws_ptr, ws_bytes, _stream_handle(stream)))

    def run_static_workspace(self, A_r, B_r, C_r, stream=None):
        """shmm_run on the library's fixed 64 MiB device workspace, for
        callers that cannot allocate device memory (see include/shmm.h)."""
        _check(lib().shmm_run_static_workspace(self._h, _ptr_array(A_r, "A"), _ptr_array(B_r, "B"),
                                               _ptr_array(C_r, "C"), _stream_handle(stream)))


# Same names as the C-ABI, for callers that prefer the flat interface.
def shmm_plan(mesh, spec_A, spec_B, spec_C, I, J, K, in_dtype="bf16", out_dtype="bf16", flags=0) -> Plan:
    return Plan(mesh, spec_A, spec_B, spec_C, I, J, K, in_dtype, out_dtype, flags)


def shmm_plan_destroy(plan: Plan) -> None:
    plan.close()


def shmm_plan_set_sm_limit(plan: Plan, max_sms: int) -> None:
    plan.set_sm_limit(max_sms)


def shmm_plan_query(plan: Plan) -> shmm_plan_info_t:
    return plan.query()


def shmm_plan_rank_box(plan: Plan, tensor: int, rank: int):
    return plan.rank_box(tensor, rank)


def shmm_workspace_size(plan: Plan) -> int:
    return plan.workspace_size()


def shmm_local_matmul(plan: Plan, A_r, B_r, P_r, stream=None):
    plan.local_matmul(A_r, B_r, P_r, stream)


def shmm_reduce_scatter(plan: Plan, P_r, C_r, stream=None):
    plan.reduce_scatter(P_r, C_r, stream)


def shmm_all_reduce(plan: Plan, P_r, C_r, stream=None):
    plan.all_reduce(P_r, C_r, stream)


def shmm_all_gather(plan: Plan, tensor: int, shard_r, full_r, stream=None):
    plan.all_gather(tensor, shard_r, full_r, stream)


def shmm_run(plan: Plan, A_r, B_r, C_r, workspace=None, stream=None):
    plan.run(A_r, B_r, C_r, workspace, stream)


def shmm_run_batch(plans: Sequence[Plan], A_r, B_r, C_r, workspaces=None, stream=None):
    """Independent sharded matmuls whose local GEMMs share launches (see
    include/shmm.h).  A_r, B_r, C_r: per plan, its list of per-rank tensors;
    workspaces: per plan, a workspace tensor or None."""
    n = len(plans)
    keep = [[_ptr_array(t, w) for t in lists] for lists, w in ((A_r, "A"), (B_r, "B"), (C_r, "C"))]
    PP = ctypes.POINTER(ctypes.c_void_p)
    tables = [(PP * n)(*[ctypes.cast(a, PP) for a in arrs]) for arrs in keep]
    ws = list(workspaces) if workspaces is not None else [None] * n
    ws_ptr = (ctypes.c_void_p * n)(*[None if w is None else w.data_ptr() for w in ws])
    ws_bytes = (ctypes.c_size_t * n)(*[0 if w is None else w.numel() * w.element_size() for w in ws])
    handles = (ctypes.c_void_p * n)(*[p.handle.value for p in plans])
    _check(lib().shmm_run_batch(n, handles, tables[0], tables[1], tables[2], ws_ptr, ws_bytes,
                                _stream_handle(stream)))


def shmm_run_host(plan: Plan, A_host, B_host, C_host, A_r, B_r, C_r, workspace=None, stream=None):
    plan.run_host(A_host, B_host, C_host, A_r, B_r, C_r, workspace, stream)


def shmm_run_static_workspace(plan: Plan, A_r, B_r, C_r, stream=None):
    plan.run_static_workspace(A_r, B_r, C_r, stream)


STATIC_WORKSPACE_BYTES = 64 << 20


def shmm_sync_status(stream=None) -> None:
    _check(lib().shmm_sync_status(_stream_handle(stream)))


def shmm_layernorm(x, gamma, beta, y, eps: float = 1e-5, stream=None):
    """Row-wise layer normalisation of a 2-D CUDA tensor x into y."""
    rows, cols = x.shape
    dt = {"torch.float32": "f32", "torch.bfloat16": "bf16"}[str(x.dtype)]
    _check(lib().shmm_layernorm(int(rows), int(cols), DTYPE_CODES[dt], x.data_ptr(), gamma.data_ptr(),
                                beta.data_ptr(), float(eps), y.data_ptr(), _stream_handle(stream)))


def shmm_reshard(mesh, spec_from, spec_to, rows: int, cols: int, dtype: str, src_r, dst_r, stream=None):
    """All-to-all / reshard of a [rows, cols] array between two shardings
    (see include/shmm.h); src_r, dst_r are per-rank tensors (or pointers)."""
    m = _mesh_struct(mesh)
    a, b = _spec_struct(mesh, spec_from), _spec_struct(mesh, spec_to)
    _check(lib().shmm_reshard(ctypes.byref(m), ctypes.byref(a), ctypes.byref(b), int(rows), int(cols),
                              DTYPE_CODES[dtype], _ptr_array(src_r, "src"), _ptr_array(dst_r, "dst"),
                              _stream_handle(stream)))


def shmm_choose_operand(B: int, D: int, F: int, axis_size: int, flops_per_s: float, bytes_per_s: float,
                        elem_bytes: int = 2) -> shmm_operand_choice_t:
    """Which operand of X[B,D].W[D_X,F] to move: 1 = all-gather W, 2 = keep W
    sharded and all-reduce the [B,F] partials (see include/shmm.h)."""
    dev = shmm_device_model_t(float(flops_per_s), float(bytes_per_s))
    out = shmm_operand_choice_t()
    _check(lib().shmm_choose_operand(int(B), int(D), int(F), int(axis_size), int(elem_bytes),
                                     ctypes.byref(dev), ctypes.byref(out)))
    return out


def shmm_selftest_wait_timeout(limit_cycles: int, stream=None) -> None:
    _check(lib().shmm_selftest_wait_timeout(int(limit_cycles), _stream_handle(stream)))


def shmm_version() -> int:
    return lib().shmm_version()


def shmm_bounds_checked() -> bool:
    """True if the loaded library is the bounds-checked build."""
    return bool(lib().shmm_bounds_checked())


def shmm_kernel_launches() -> int:
    return lib().shmm_kernel_launches()
