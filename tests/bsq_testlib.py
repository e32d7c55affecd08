"""Shared helpers of the test suite (not a test module)."""
from __future__ import annotations

import numpy as np

SENTINEL = 0xA5
MARGIN = 256


def to_device_bf16(bits: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def u32_device(a: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint32).view(np.int32)).to(device)


def i32_device(a: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def guarded(nbytes: int, device="cuda"):
    """A uint8 device buffer of nbytes plus a sentinel-filled margin: returns
    (full buffer, view of the first nbytes)."""
    import torch
    full = torch.full((nbytes + MARGIN,), SENTINEL, dtype=torch.uint8, device=device)
    return full, full[:nbytes]


def margin_intact(full) -> bool:
    tail = full[-MARGIN:].cpu().numpy()
    return bool(np.all(tail == SENTINEL))
