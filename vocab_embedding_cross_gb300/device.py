"""Moves seeded host arrays to the GPU as torch tensors (plumbing only).

bf16 inputs arrive as uint16 bit patterns and are reinterpreted, not
converted, so the device holds exactly the values the oracle reads.
"""
from __future__ import annotations

import numpy as np
import torch


def to_device(arr: np.ndarray, device="cuda", pin: bool = False) -> torch.Tensor:
    if arr.dtype == np.uint16:
        t = torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr))
    if pin:
        t = t.pin_memory()
    return t.to(device, non_blocking=pin)


def to_host_bits(t: torch.Tensor) -> np.ndarray:
    """Device tensor back to numpy; bf16 comes back as uint16 bit patterns."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A 256-byte aligned uint8 workspace (the caching allocator aligns to 512)."""
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)
