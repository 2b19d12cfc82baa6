"""Moves seeded workloads into torch tensors (host or device).  Layout only, no arithmetic."""
from __future__ import annotations

import numpy as np
import torch


def tensor(arr: np.ndarray, dtype: str, device=None, pin: bool = False) -> torch.Tensor:
    """numpy array (uint16 bf16 bits or fp32) -> torch tensor of the stored dtype."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32))
    if pin:
        t = t.pin_memory()
    return t.to(device) if device is not None else t


def index(arr: np.ndarray, device=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.uint32).view(np.int32))
    return t.to(device) if device is not None else t


def prefill_inputs(p, device) -> dict:
    """Device tensors of a workloads.Problem, keyed like kda.prefill's arguments."""
    return dict(q=tensor(p.q, p.qkv_dtype, device), k=tensor(p.k, p.qkv_dtype, device),
                v=tensor(p.v, p.qkv_dtype, device), beta=tensor(p.beta, "f32", device),
                log_decay=tensor(p.g, "f32", device),
                input_row_offsets=index(p.offsets, device), slot_idx=index(p.slot_idx, device),
                state_pool=tensor(p.pool, p.state_dtype, device))


def decode_inputs(dp, device) -> dict:
    """Device tensors of a workloads.DecodeProblem: per-step inputs stacked on dim 0."""
    return dict(q=tensor(dp.q, dp.qkv_dtype, device), k=tensor(dp.k, dp.qkv_dtype, device),
                v=tensor(dp.v, dp.qkv_dtype, device), beta=tensor(dp.beta, "f32", device),
                log_decay=tensor(dp.g, "f32", device), slot_idx=index(dp.slot_idx, device),
                state_pool=tensor(dp.pool, dp.state_dtype, device))


def pool_to_f64(pool: torch.Tensor) -> np.ndarray:
    return pool.detach().float().cpu().numpy().astype(np.float64)
