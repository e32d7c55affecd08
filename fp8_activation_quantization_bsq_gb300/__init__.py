"""Block-scaled BF16 -> NVFP4 / MXFP4 / MXFP8 quantization for NVIDIA GB300.

Thin Python binding of ``libbsq`` (C ABI in ``include/bsq.h``): it turns
torch tensors into pointers and sizes, allocates missing outputs with torch,
passes torch's current CUDA stream and raises on a non-zero status.  Every
step of the computation runs in the library's CUDA kernels; there is no CPU
path.  The binding fails loudly when ``libbsq.so`` has not been built
(``python -m fp8_activation_quantization_bsq_gb300._build`` or
``__graft_entry__.build()``).

Operations (Modular "block_scaled_quantization" pages):
  quantize            -- quantize_dynamic_block_scaled / quantize_dynamic_scaled_fp4fp8
  grouped_quantize    -- grouped_quantize_dynamic_scaled_fp4_async(_kernel)
  scales_interleave   -- block_scales_interleave(_fp4)(_kernel)
  block_scaled_dot    -- the idea of naive_block_scaled_matmul (a validator)
and the steps around them: tensor_sf / grouped_tensor_sf (the NVFP4 tensor
scales on the GPU), quantize_dynamic (tensor_sf read from device memory),
grouped_quantize_dynamic (per-expert scales on the GPU, then the grouped
quantize), gemm_quantize (a matmul with the quantize in its epilogue).
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB_PATH

__all__ = ["FORMATS", "GROUPED_KERNELS", "lib", "BsqError", "block_size", "packed_row_bytes",
           "scales5d_bytes", "quantize", "quantize_dynamic", "tensor_sf", "grouped_tensor_sf",
           "grouped_quantize_dynamic",
           "grouped_quantize", "grouped_quantize_workspace_bytes", "scales_interleave", "block_scaled_dot", "gemm_quantize", "device_error",
           "status_string"]

FORMATS = {"nvfp4": 0, "mxfp4": 1, "mxfp8": 2}
GROUPED_KERNELS = {"auto": 0, "stream": 1, "latency": 2, "token": 3}

_c_i32, _c_i64, _c_f32, _c_p = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p

_SIGNATURES = {
    "bsq_version": (_c_i32, []),
    "bsq_status_string": (ctypes.c_char_p, [_c_i32]),
    "bsq_block_size": (_c_i32, [_c_i32]),
    "bsq_packed_row_bytes": (_c_i64, [_c_i32, _c_i64]),
    "bsq_scales5d_bytes": (_c_i64, [_c_i32, _c_i64, _c_i64]),
    "bsq_quantize": (_c_i32, [_c_i32, _c_p, _c_i64, _c_i64, _c_i64, _c_p, _c_p, _c_f32, _c_p]),
    "bsq_grouped_quantize": (_c_i32, [_c_i32, _c_p, _c_i64, _c_i64, _c_i64, _c_p, _c_p, _c_p,
                                      _c_p, _c_i32, _c_p, _c_i32, _c_i64, _c_i64, _c_p, _c_p,
                                      _c_i32, _c_p]),
    "bsq_grouped_quantize_kernel": (_c_i32, [_c_i32, _c_p, _c_i64, _c_i64, _c_i64, _c_p, _c_p,
                                             _c_p, _c_p, _c_i32, _c_p, _c_i32, _c_i64, _c_i64,
                                             _c_p, _c_p, _c_i32, _c_i32, _c_p]),
    "bsq_grouped_quantize_workspace_bytes": (_c_i64, [_c_i32, _c_i64, _c_i64]),
    "bsq_grouped_quantize_ws": (_c_i32, [_c_i32, _c_p, _c_i64, _c_i64, _c_i64, _c_p, _c_p,
                                         _c_p, _c_p, _c_i32, _c_p, _c_i32, _c_i64, _c_i64,
                                         _c_p, _c_p, _c_i32, _c_i32, _c_p, _c_i64, _c_p]),
    "bsq_scales_interleave": (_c_i32, [_c_p, _c_i64, _c_i64, _c_i64, _c_p, _c_p]),
    "bsq_quantize_dynamic": (_c_i32, [_c_i32, _c_p, _c_i64, _c_i64, _c_i64, _c_p, _c_p, _c_p, _c_p]),
    "bsq_tensor_sf_workspace_bytes": (_c_i64, []),
    "bsq_tensor_sf": (_c_i32, [_c_p, _c_i64, _c_i64, _c_i64, _c_p, _c_p, _c_i64, _c_p]),
    "bsq_grouped_tensor_sf_workspace_bytes": (_c_i64, [_c_i32]),
    "bsq_grouped_tensor_sf_noalloc": (_c_i32, [_c_p, _c_i64, _c_i64, _c_i64, _c_p, _c_p, _c_p, _c_i32,
                                               _c_i64, _c_p, _c_i32, _c_p]),
    "bsq_grouped_tensor_sf": (_c_i32, [_c_p, _c_i64, _c_i64, _c_i64, _c_p, _c_p, _c_p, _c_i32,
                                       _c_i64, _c_p, _c_i32, _c_p, _c_i64, _c_p]),
    "bsq_device_error": (_c_i32, [_c_p, ctypes.POINTER(_c_i32)]),
    "bsq_selftest_wait_timeout": (_c_i32, [_c_p]),
    "bsq_block_scaled_dot": (_c_i32, [_c_i32, _c_p, _c_p, ctypes.c_float, _c_p, _c_p, ctypes.c_float,
                                      _c_i64, _c_i64, _c_i64, _c_p, _c_p]),
    "bsq_gemm_quantize": (_c_i32, [_c_i32, _c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_f32,
                                   _c_p, _c_p, _c_p, _c_p]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded ``libbsq.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libbsq is not built ({LIB_PATH} missing); build it with "
                               "python -m fp8_activation_quantization_bsq_gb300._build")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


class BsqError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)}")
        self.code = code


def status_string(code: int) -> str:
    return lib().bsq_status_string(code).decode()


def _check(code: int, what: str) -> None:
    if code != 0:
        raise BsqError(code, what)


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def block_size(fmt) -> int:
    return lib().bsq_block_size(_fmt(fmt))


def packed_row_bytes(fmt, K: int) -> int:
    return lib().bsq_packed_row_bytes(_fmt(fmt), K)


def scales5d_bytes(fmt, rows: int, K: int) -> int:
    return lib().bsq_scales5d_bytes(_fmt(fmt), rows, K)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(device, stream):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def quantize(x: torch.Tensor, fmt, tensor_sf: float = 1.0, out=None, scales=None, stream=None):
    """Quantize an (M, K) BF16 CUDA tensor (unit inner stride).

    Returns (packed uint8 (M, packed_row_bytes), scales uint8 [scales5d_bytes])
    with the scales in the 5D TCGEN layout.
    """
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_cuda or (x.shape[1] > 1 and x.stride(1) != 1):
        raise ValueError("x must be a 2-D bfloat16 CUDA tensor with unit inner stride")
    f = _fmt(fmt)
    M, K = x.shape
    if out is None:
        out = torch.empty((M, packed_row_bytes(f, K)), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(scales5d_bytes(f, M, K), dtype=torch.uint8, device=x.device)
    with torch.cuda.device(x.device):
        rc = lib().bsq_quantize(f, _ptr(x), M, K, x.stride(0) if M else K, _ptr(out), _ptr(scales),
                                float(tensor_sf), _stream(x.device, stream))
    _check(rc, "bsq_quantize")
    return out, scales


def quantize_dynamic(x: torch.Tensor, fmt, tensor_sf_dev=None, out=None, scales=None, stream=None):
    """Like ``quantize`` with the NVFP4 tensor_sf read from device memory
    (``tensor_sf_dev``: a float32 CUDA tensor whose first element is used,
    e.g. ``tensor_sf(x)[1:]``).  When it is None (NVFP4), the scale is computed
    first on the GPU with ``tensor_sf``; nothing waits for the host."""
    _check_x(x)
    f = _fmt(fmt)
    M, K = x.shape
    if f == FORMATS["nvfp4"] and tensor_sf_dev is None:
        tensor_sf_dev = tensor_sf(x, stream=stream)[1:]
    if out is None:
        out = torch.empty((M, packed_row_bytes(f, K)), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(scales5d_bytes(f, M, K), dtype=torch.uint8, device=x.device)
    with torch.cuda.device(x.device):
        rc = lib().bsq_quantize_dynamic(f, _ptr(x), M, K, x.stride(0) if M else K, _ptr(out),
                                        _ptr(scales), _ptr(tensor_sf_dev), _stream(x.device, stream))
    _check(rc, "bsq_quantize_dynamic")
    return out, scales


def tensor_sf(x: torch.Tensor, out=None, workspace=None, stream=None):
    """float32 CUDA tensor [amax, tensor_sf] of a 2-D BF16 CUDA tensor,
    tensor_sf = fl32(448*6/amax) (1.0 for an all-zero tensor).  A reused
    ``workspace`` must have been zeroed once (``torch.zeros``); each call
    leaves it zeroed."""
    _check_x(x)
    M, K = x.shape
    if out is None:
        out = torch.empty(2, dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.zeros(lib().bsq_tensor_sf_workspace_bytes(), dtype=torch.uint8, device=x.device)
    with torch.cuda.device(x.device):
        rc = lib().bsq_tensor_sf(_ptr(x), M, K, x.stride(0) if M else K, _ptr(out), _ptr(workspace),
                                 workspace.numel(), _stream(x.device, stream))
    _check(rc, "bsq_tensor_sf")
    return out


def grouped_tensor_sf(x: torch.Tensor, row_offsets, expert_ids, num_experts: int,
                      row_indices=None, total_rows: int | None = None, out=None, workspace=None,
                      stream=None):
    """float32 CUDA tensor [num_experts] of per-expert tensor scales over the
    experts' gathered rows (1.0 for experts without rows)."""
    _check_x(x)
    in_rows, K = x.shape
    G = expert_ids.numel()
    if total_rows is None:
        total_rows = row_indices.numel() if row_indices is not None else in_rows
    if out is None:
        out = torch.empty(num_experts, dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.zeros(lib().bsq_grouped_tensor_sf_workspace_bytes(num_experts),
                                dtype=torch.uint8, device=x.device)
    with torch.cuda.device(x.device):
        rc = lib().bsq_grouped_tensor_sf(_ptr(x), in_rows, K, x.stride(0) if in_rows else K,
                                         _ptr(row_offsets), _ptr(expert_ids), _ptr(row_indices), G,
                                         total_rows, _ptr(out), num_experts, _ptr(workspace),
                                         workspace.numel(), _stream(x.device, stream))
    _check(rc, "bsq_grouped_tensor_sf")
    return out


def _check_x(x):
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_cuda or (x.shape[1] > 1 and x.stride(1) != 1):
        raise ValueError("x must be a 2-D bfloat16 CUDA tensor with unit inner stride")


def grouped_quantize(x: torch.Tensor, fmt, row_offsets, scales_offsets, expert_ids,
                     sf_tensor=None, row_indices=None, total_rows: int | None = None,
                     total_scale_rows: int | None = None, k_tiles_per_block: int = 1,
                     out=None, scales=None, stream=None, kernel: str = "auto", workspace=None):
    """Grouped per-expert quantize of the (in_rows, K) BF16 CUDA tensor ``x``.

    ``row_offsets`` / ``scales_offsets`` are uint32 (stored as torch.int32
    bit patterns or uint32) CUDA tensors of G+1 entries, ``expert_ids`` int32
    [G], ``sf_tensor`` float32 [num_experts] (NVFP4), ``row_indices`` int32 or
    None.  ``total_rows`` / ``total_scale_rows`` size the outputs (required
    when ``out`` / ``scales`` are not given).  ``kernel``: "auto", "stream"
    (groups of many rows), "latency" (groups of a few rows) or "token" (a
    row_indices gather that reuses source rows: each read once); the results
    do not depend on it.  ``k_tiles_per_block``: 1, 2, 4, 8, or 0 (chosen by
    the library).  ``workspace``: None, or a CUDA uint8 tensor of at least
    ``grouped_quantize_workspace_bytes(fmt, total_scale_rows, K)`` bytes in
    which the token kernel stages NVFP4 scale rows (same results; in use
    until the call's work on the stream completes; MX formats ignore it).
    Returns (packed uint8 (total_rows, packed_row_bytes), scales uint8).
    """
    if kernel not in GROUPED_KERNELS:
        raise ValueError(f"kernel must be one of {sorted(GROUPED_KERNELS)}")
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_cuda or (x.shape[1] > 1 and x.stride(1) != 1):
        raise ValueError("x must be a 2-D bfloat16 CUDA tensor with unit inner stride")
    f = _fmt(fmt)
    in_rows, K = x.shape
    G = expert_ids.numel()
    if total_rows is None:
        if out is None:
            raise ValueError("total_rows is required when out is not given")
        total_rows = out.shape[0]
    if total_scale_rows is None:
        raise ValueError("total_scale_rows is required")
    if out is None:
        out = torch.empty((total_rows, packed_row_bytes(f, K)), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(scales5d_bytes(f, total_scale_rows, K), dtype=torch.uint8, device=x.device)
    num_experts = sf_tensor.numel() if sf_tensor is not None else 0
    with torch.cuda.device(x.device):
        rc = lib().bsq_grouped_quantize_ws(
            f, _ptr(x), in_rows, K, x.stride(0) if in_rows else K, _ptr(row_offsets),
            _ptr(scales_offsets), _ptr(expert_ids), _ptr(sf_tensor), num_experts,
            _ptr(row_indices), G, total_rows, total_scale_rows, _ptr(out), _ptr(scales),
            k_tiles_per_block, GROUPED_KERNELS[kernel], _ptr(workspace),
            workspace.numel() * workspace.element_size() if workspace is not None else 0,
            _stream(x.device, stream))
    _check(rc, "bsq_grouped_quantize")
    return out, scales


def grouped_quantize_dynamic(x: torch.Tensor, row_offsets, scales_offsets, expert_ids, num_experts: int,
                             row_indices=None, total_rows: int | None = None,
                             total_scale_rows: int | None = None, k_tiles_per_block: int = 0,
                             out=None, scales=None, sf_out=None, tsf_workspace=None, workspace=None,
                             stream=None, kernel: str = "auto"):
    """Grouped NVFP4 quantize with the per-expert tensor scales computed on
    the GPU first (``grouped_tensor_sf``) and read by the quantize from
    device memory, both on one stream with nothing waiting for the host.
    ``tsf_workspace``: the scales' reduction workspace (zeroed once, left
    zeroed; allocated when None); ``workspace``: as for
    :func:`grouped_quantize`.  Returns (packed, scales, sf_tensor
    float32 [num_experts])."""
    if total_rows is None:
        if out is None:
            raise ValueError("total_rows is required when out is not given")
        total_rows = out.shape[0]
    sf = grouped_tensor_sf(x, row_offsets, expert_ids, num_experts, row_indices, total_rows=total_rows,
                           out=sf_out, workspace=tsf_workspace, stream=stream)
    packed, sc = grouped_quantize(x, "nvfp4", row_offsets, scales_offsets, expert_ids, sf, row_indices,
                                  total_rows=total_rows, total_scale_rows=total_scale_rows,
                                  k_tiles_per_block=k_tiles_per_block, out=out, scales=scales, stream=stream,
                                  kernel=kernel, workspace=workspace)
    return packed, sc, sf


def grouped_quantize_workspace_bytes(fmt, total_scale_rows: int, K: int) -> int:
    """Bytes of the ``workspace`` of :func:`grouped_quantize`."""
    return int(lib().bsq_grouped_quantize_workspace_bytes(_fmt(fmt), total_scale_rows, K))


def scales_interleave(scales2d: torch.Tensor, out=None, stream=None):
    """Rank-2 (M, S) uint8 CUDA scales (unit inner stride) -> 5D layout."""
    if scales2d.dtype != torch.uint8 or scales2d.dim() != 2 or not scales2d.is_cuda or \
            (scales2d.shape[1] > 1 and scales2d.stride(1) != 1):
        raise ValueError("scales2d must be a 2-D uint8 CUDA tensor with unit inner stride")
    M, S = scales2d.shape
    if out is None:
        nbytes = -(-M // 128) * -(-S // 4) * 512
        out = torch.empty(nbytes, dtype=torch.uint8, device=scales2d.device)
    with torch.cuda.device(scales2d.device):
        rc = lib().bsq_scales_interleave(_ptr(scales2d), M, S, scales2d.stride(0) if M else S,
                                         _ptr(out), _stream(scales2d.device, stream))
    _check(rc, "bsq_scales_interleave")
    return out


def block_scaled_dot(fmt, a_packed: torch.Tensor, a_scales: torch.Tensor, b_packed: torch.Tensor,
                     b_scales: torch.Tensor, K: int, a_tsf: float = 1.0, b_tsf: float = 1.0,
                     out=None, stream=None) -> torch.Tensor:
    """float64 (M, N) = dequantized A (M, K) times dequantized B (N, K)^T, from
    packed rows and 5D scales (a slow FP64 validator, not a fast matmul)."""
    f = _fmt(fmt)
    M, N = a_packed.shape[0], b_packed.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float64, device=a_packed.device)
    with torch.cuda.device(a_packed.device):
        rc = lib().bsq_block_scaled_dot(f, _ptr(a_packed), _ptr(a_scales), float(a_tsf), _ptr(b_packed),
                                        _ptr(b_scales), float(b_tsf), M, N, K, _ptr(out),
                                        _stream(a_packed.device, stream))
    _check(rc, "bsq_block_scaled_dot")
    return out


def gemm_quantize(a: torch.Tensor, b: torch.Tensor, fmt, tensor_sf: float = 1.0, out=None, scales=None,
                  c_out=None, stream=None):
    """C = a (M, K) @ b (N, K)^T in BF16 with FP32 accumulation, quantized in
    the matmul's epilogue: returns (packed uint8 (M, packed_row_bytes(N)),
    scales uint8 [scales5d_bytes(M, N)]) as ``quantize`` would give for the
    BF16 C, which is not stored unless ``c_out`` (a (M, N) bfloat16 CUDA
    tensor) is given.  N % 128 == 0, K % 32 == 0."""
    for t in (a, b):
        if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_cuda or (t.shape[1] > 1 and t.stride(1) != 1):
            raise ValueError("a and b must be 2-D bfloat16 CUDA tensors with unit inner stride")
    if a.shape[1] != b.shape[1]:
        raise ValueError("a and b must have the same K")
    f = _fmt(fmt)
    M, K = a.shape
    N = b.shape[0]
    if out is None:
        out = torch.empty((M, packed_row_bytes(f, N)), dtype=torch.uint8, device=a.device)
    if scales is None:
        scales = torch.empty(scales5d_bytes(f, M, N), dtype=torch.uint8, device=a.device)
    if c_out is not None and (c_out.dtype != torch.bfloat16 or tuple(c_out.shape) != (M, N) or
                              not c_out.is_contiguous()):
        raise ValueError("c_out must be a contiguous (M, N) bfloat16 tensor")
    with torch.cuda.device(a.device):
        rc = lib().bsq_gemm_quantize(f, _ptr(a), _ptr(b), M, N, K, a.stride(0) if M else K,
                                     b.stride(0) if N else K, float(tensor_sf), _ptr(out), _ptr(scales),
                                     _ptr(c_out), _stream(a.device, stream))
    _check(rc, "bsq_gemm_quantize")
    return out, scales


def device_error(device=None, stream=None) -> int:
    """Synchronize and read-and-clear the device's error word (0 = none)."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    code = _c_i32(0)
    with torch.cuda.device(device):
        rc = lib().bsq_device_error(_stream(device, stream), ctypes.byref(code))
    _check(rc, "bsq_device_error")
    return code.value
