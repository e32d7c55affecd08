"""Block-scaled quantization steps (oracle; test infrastructure only).

Follows the NVFP4 kernel page (quantize_dynamic_scaled_async_fp4_kernel,
description and signature: one scale per group of SF_VECTOR_SIZE elements,
FP4 codes packed two per byte, an FP32 ``tensor_sf`` argument), the three
formats named on the block_scaled_quantization module page, and the grouped
kernel's arguments (grouped_quantize_dynamic_scaled_fp4_async_kernel,
signature), under the readings stated in the package header.
"""
from __future__ import annotations

import numpy as np

from .formats import (e2m1_encode, e4m3_encode, e2m1_decode, e4m3_decode,
                      e8m0_decode, e8m0_ceil_exponent)
from .layout import offset_5d, scales_to_5d, scales5d_bytes

FORMATS = ("nvfp4", "mxfp4", "mxfp8")


def block_size(fmt: str) -> int:
    """Elements per scale factor: 16 for NVFP4, 32 for MXFP4 / MXFP8."""
    return {"nvfp4": 16, "mxfp4": 32, "mxfp8": 32}[fmt]


def packed_row_bytes(fmt: str, K: int) -> int:
    """Bytes of one packed output row: K/2 for the 4-bit formats, K for MXFP8."""
    return K if fmt == "mxfp8" else K // 2


def _bf16_to_f32(x_bits: np.ndarray) -> np.ndarray:
    return (np.asarray(x_bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def nvfp4_block_scale(amax: np.ndarray, tsf: np.float32) -> np.ndarray:
    """NVFP4 block scale byte: E4M3(fl32(fl32(amax / 6) * tensor_sf))."""
    with np.errstate(over="ignore"):                 # +inf saturates to 448
        s = (np.asarray(amax, np.float32) / np.float32(6.0)) * np.float32(tsf)
    return e4m3_encode(s)


def nvfp4_element_scale(scale_bytes: np.ndarray, tsf: np.float32) -> np.ndarray:
    """NVFP4 element scale: 0 when the decoded block scale ds is 0, else
    fl32(tensor_sf / ds)."""
    ds = e4m3_decode(scale_bytes).astype(np.float32)
    safe = np.where(ds == 0, np.float32(1.0), ds)
    return np.where(ds == 0, np.float32(0.0), np.float32(tsf) / safe).astype(np.float32)


def mx_block_exponent(amax: np.ndarray, qmax: float) -> np.ndarray:
    """MX block exponent e: ceil(log2(fl32(amax / Qmax))) clamped to
    [-127, 127]; -127 for an all-zero block.  The scale byte is e + 127."""
    s = np.asarray(amax, np.float32) / np.float32(qmax)
    return np.where(s == 0, -127, np.clip(e8m0_ceil_exponent(s), -127, 127)).astype(np.int64)


def quantize_rank2(fmt: str, x_bits: np.ndarray, tensor_sf=1.0):
    """Quantize an (M, K) BF16 matrix (uint16 bits).

    Returns (packed uint8 (M, packed_row_bytes), scales uint8 (M, K/SF)),
    scales in plain row-major (rank-2) order.
    """
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    M, K = x_bits.shape
    SF = block_size(fmt)
    assert K % SF == 0
    S = K // SF
    blocks = _bf16_to_f32(x_bits).reshape(M, S, SF)
    amax = np.abs(blocks).max(axis=-1) if S else np.zeros((M, 0), np.float32)

    if fmt == "nvfp4":
        tsf = np.float32(tensor_sf)
        scale_bytes = nvfp4_block_scale(amax, tsf)
        factor = nvfp4_element_scale(scale_bytes, tsf)
        with np.errstate(over="ignore"):             # +-inf saturates to +-6
            codes = e2m1_encode(blocks * factor[..., None])
    else:
        e = mx_block_exponent(amax, 6.0 if fmt == "mxfp4" else 448.0)
        scale_bytes = (e + 127).astype(np.uint8)
        factor = np.ldexp(np.float64(1.0), -e).astype(np.float32)   # 2^-e, exact in FP32
        y = blocks * factor[..., None]
        codes = e2m1_encode(y) if fmt == "mxfp4" else e4m3_encode(y)

    codes = codes.reshape(M, K)
    if fmt == "mxfp8":
        packed = codes.astype(np.uint8)
    else:
        packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, scale_bytes.astype(np.uint8).reshape(M, S)


def quantize(fmt: str, x_bits: np.ndarray, tensor_sf=1.0):
    """Dense quantize: (packed (M, row bytes), scales in the zero-padded 5D layout)."""
    packed, scales = quantize_rank2(fmt, x_bits, tensor_sf)
    return packed, scales_to_5d(scales)


def grouped_quantize(fmt: str, x_bits: np.ndarray, row_offsets, scales_offsets,
                     expert_ids, sf_tensor=None, row_indices=None,
                     total_rows: int | None = None, total_scale_rows: int | None = None):
    """Grouped per-expert quantize.

    Group g (expert ``expert_ids[g]``; skipped when negative) owns destination
    rows ``row_offsets[g] .. row_offsets[g+1]-1`` and scale rows starting at
    ``scales_offsets[g]``.  Local row i reads source row
    ``row_indices[row_offsets[g]+i]`` (or ``row_offsets[g]+i`` without
    ``row_indices``), is quantized with tensor_sf = ``sf_tensor[expert]``
    (NVFP4), written to packed row ``row_offsets[g]+i`` and its scales to 5D
    row ``scales_offsets[g]+i`` (all Kt*4 columns, padding columns 0).

    Returns (packed, packed_row_written, scales5d, scales5d_written).
    """
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    K = x_bits.shape[1]
    ro = np.asarray(row_offsets, dtype=np.int64)
    so = np.asarray(scales_offsets, dtype=np.int64)
    eid = np.asarray(expert_ids, dtype=np.int64)
    G = eid.size
    SF = block_size(fmt)
    S = K // SF
    Kt = -(-S // 4)
    if total_rows is None:
        total_rows = int(ro[G]) if G else 0
    if total_scale_rows is None:
        total_scale_rows = int(so[G]) if G else 0
    packed = np.zeros((total_rows, packed_row_bytes(fmt, K)), dtype=np.uint8)
    row_written = np.zeros(total_rows, dtype=bool)
    scales = np.zeros(scales5d_bytes(total_scale_rows, S), dtype=np.uint8)
    scales_written = np.zeros(scales.size, dtype=bool)
    for g in range(G):
        if eid[g] < 0:
            continue
        rows = np.arange(ro[g], ro[g + 1])
        src = np.asarray(row_indices, dtype=np.int64)[rows] if row_indices is not None else rows
        tsf = np.float32(sf_tensor[eid[g]]) if fmt == "nvfp4" else np.float32(1.0)
        p, sc = quantize_rank2(fmt, x_bits[src], tsf)
        packed[rows] = p
        row_written[rows] = True
        full = np.zeros((rows.size, Kt * 4), dtype=np.uint8)
        full[:, :S] = sc
        srow = so[g] + np.arange(rows.size)
        m, s = np.meshgrid(srow, np.arange(Kt * 4), indexing="ij")
        off = offset_5d(m, s, Kt)
        scales[off] = full
        scales_written[off] = True
    return packed, row_written, scales, scales_written


def dequantize(fmt: str, packed: np.ndarray, scales2d: np.ndarray, tensor_sf=1.0) -> np.ndarray:
    """Decode packed codes times their block scale (float64, (M, K))."""
    packed = np.asarray(packed, dtype=np.uint8)
    M = packed.shape[0]
    if fmt == "mxfp8":
        vals = e4m3_decode(packed)
    else:
        codes = np.empty((M, packed.shape[1] * 2), dtype=np.uint8)
        codes[:, 0::2] = packed & 0xF
        codes[:, 1::2] = packed >> 4
        vals = e2m1_decode(codes)
    K = vals.shape[1]
    SF = block_size(fmt)
    sc = np.asarray(scales2d, dtype=np.uint8)[:M, : K // SF]
    if fmt == "nvfp4":
        factor = e4m3_decode(sc) / np.float64(np.float32(tensor_sf))
    else:
        factor = e8m0_decode(sc)
    return vals * np.repeat(factor, SF, axis=1)
