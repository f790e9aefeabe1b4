"""shmm: GB300-native sharded matmul A[I,J].B[J,K] -> C[I,K] with the
partial-sum reduction its sharding requires, for virtual ranks held on one
GPU.  The compute lives in libshmm.so (hand-written sm_103a CUDA behind the
C-ABI of include/shmm.h); this package is its Python binding and build."""
from .shmm import (  # noqa: F401
    BF16, F32, FLAG_FUSED, FLAG_GELU, FLAG_PARTIAL_OUT_DTYPE, FLAG_RANK_ORDER, FLAG_SIMT, FLAG_TREE, Plan,
    ShmmError, TENSOR_A, TENSOR_A_LOCAL, TENSOR_B, TENSOR_B_LOCAL, TENSOR_C, TENSOR_C_REDUCED, TENSOR_P, lib,
    parse_mesh, parse_spec, shmm_all_gather, shmm_all_reduce, shmm_bounds_checked, shmm_choose_operand,
    shmm_kernel_launches, shmm_layernorm, shmm_local_matmul, shmm_plan, shmm_plan_destroy, shmm_plan_query,
    shmm_plan_rank_box, shmm_plan_set_sm_limit, shmm_reduce_scatter, shmm_reshard, shmm_run, shmm_run_batch,
    shmm_run_host, shmm_selftest_wait_timeout, shmm_sync_status, shmm_version, shmm_workspace_size)
from . import helpers  # noqa: F401
