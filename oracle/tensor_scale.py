"""Per-tensor and per-expert NVFP4 tensor scales (oracle; test infrastructure only).

The NVFP4 kernel takes an FP32 ``tensor_sf`` (quantize_dynamic_scaled_async_fp4_kernel
signature) and the grouped kernel one FP32 scale per expert in ``sf_tensor``
(grouped_quantize_dynamic_scaled_fp4_async_kernel, argument list).  Reading: ``tensor_sf = fl32(448 * 6 / amax)`` with amax the exact
max |x| over the tensor (over the expert's gathered rows), 1.0 for an all-zero
tensor, so that the largest block maps onto the E4M3 maximum 448.
"""
from __future__ import annotations

import numpy as np


def _amax(x_bits: np.ndarray) -> np.float32:
    b = np.asarray(x_bits, dtype=np.uint16)
    if b.size == 0:
        return np.float32(0.0)
    mags = (b.astype(np.uint32) & 0x7FFF) << 16        # |x| as FP32 bit patterns
    return np.uint32(mags.max()).view(np.float32)


def tensor_sf(x_bits: np.ndarray):
    """(amax, tensor_sf) of a BF16 tensor (uint16 bits), both FP32."""
    amax = _amax(x_bits)
    if amax == 0:
        return amax, np.float32(1.0)
    with np.errstate(over="ignore"):
        return amax, np.float32(np.float32(2688.0) / amax)


def expert_tensor_sf(x_bits, row_offsets, expert_ids, num_experts: int, row_indices=None):
    """Per-expert (amax[num_experts], sf[num_experts]): amax over the rows of
    every group of the expert (sources via row_indices), sf as in
    ``tensor_sf``; experts without rows get amax 0 and sf 1.0."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    ro = np.asarray(row_offsets, dtype=np.int64)
    eid = np.asarray(expert_ids, dtype=np.int64)
    amax = np.zeros(num_experts, dtype=np.float32)
    for g, e in enumerate(eid):
        if e < 0:
            continue
        rows = np.arange(ro[g], ro[g + 1])
        src = np.asarray(row_indices, dtype=np.int64)[rows] if row_indices is not None else rows
        amax[e] = max(amax[e], _amax(x_bits[src]))
    sf = np.ones(num_experts, dtype=np.float32)
    nz = amax > 0
    with np.errstate(over="ignore"):
        sf[nz] = np.float32(2688.0) / amax[nz]
    return amax, sf
