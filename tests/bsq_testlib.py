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


def _oracle_rank2_job(job):
    """Process-pool task: the oracle's quantize_rank2 of one chunk of rows."""
    import oracle
    fmt, bits, tsf = job
    return oracle.quantize_rank2(fmt, bits, tsf)


def oracle_rank2_chunks(fmt, jobs):
    """oracle.quantize_rank2 over a list of (bits, tsf) jobs, spread over a
    spawned process pool (one worker per host core): [(packed, scales2d)]."""
    import multiprocessing as mp
    import os
    from concurrent.futures import ProcessPoolExecutor
    with ProcessPoolExecutor(max_workers=max(1, os.cpu_count() or 1), mp_context=mp.get_context("spawn")) as pool:
        return list(pool.map(_oracle_rank2_job, [(fmt, b, t) for b, t in jobs], chunksize=1))
