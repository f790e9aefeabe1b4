"""Per-rank buffer helpers for the binding: allocate a plan's per-rank boxes,
cut a global host array into them, or read them back.  Data movement only;
none of the method's arithmetic."""
from __future__ import annotations

from typing import List, Optional

import torch

from .shmm import F32, TENSOR_P, Plan

TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def tensor_dtype(plan: Plan, tensor: int) -> torch.dtype:
    """dtype of a plan's buffers of kind ``tensor``."""
    from .shmm import TENSOR_A, TENSOR_A_LOCAL, TENSOR_B, TENSOR_B_LOCAL
    if tensor in (TENSOR_A, TENSOR_B, TENSOR_A_LOCAL, TENSOR_B_LOCAL):
        return TORCH_DTYPES[plan.in_dtype]
    if tensor == TENSOR_P and plan.info.collective != 0:
        return torch.float32 if plan.info.partial_dtype == F32 else torch.bfloat16
    return TORCH_DTYPES[plan.out_dtype]


def alloc(plan: Plan, tensor: int, device="cuda", dtype: Optional[torch.dtype] = None,
          fill: Optional[float] = None) -> List[torch.Tensor]:
    """One dense buffer per rank holding the rank's box of ``tensor``."""
    dt = dtype or tensor_dtype(plan, tensor)
    out = []
    for r in range(plan.nranks):
        _, ext = plan.rank_box(tensor, r)
        t = torch.empty(ext, dtype=dt, device=device)
        if fill is not None:
            t.fill_(fill)
        out.append(t)
    return out


def shard(plan: Plan, tensor: int, full: torch.Tensor, device="cuda") -> List[torch.Tensor]:
    """Each rank's box of the global array ``full`` as its own contiguous
    device buffer (replicated blocks are copied once per rank)."""
    out = []
    for r in range(plan.nranks):
        (o0, o1), (e0, e1) = plan.rank_box(tensor, r)
        out.append(full[o0:o0 + e0, o1:o1 + e1].contiguous().to(device, non_blocking=True))
    return out


def boxes(plan: Plan, tensor: int):
    return [plan.rank_box(tensor, r) for r in range(plan.nranks)]


def workspace(plan: Plan, device="cuda") -> Optional[torch.Tensor]:
    n = plan.workspace_size()
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device)
