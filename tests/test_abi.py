"""The C ABI boundary, checked on the CPU (no compute call reaches CUDA).

libbsq must load, export exactly what include/bsq.h declares, size its
buffers like the oracle's layout, and reject every bad argument with the
documented status before anything is enqueued.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bsq.h")

OK, NULL, SHAPE, ALIGN, VALUE = 0, 1, 2, 3, 4
P = 0x10000  # a fake, 16-byte aligned, never dereferenced "device" pointer


@pytest.fixture(scope="module")
def lib():
    from fp8_activation_quantization_bsq_gb300 import _build
    _build.build()
    import fp8_activation_quantization_bsq_gb300 as bsq
    return bsq.lib()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^BSQ_API\s+[\w\s\*]+?\b(bsq_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("bsq_quantize", "bsq_grouped_quantize", "bsq_scales_interleave",
              "bsq_status_string", "bsq_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    # and nothing else with the bsq_ prefix
    import subprocess
    from fp8_activation_quantization_bsq_gb300._build import LIB_PATH
    nm = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True, text=True)
    if nm.returncode == 0:
        exported = sorted(set(re.findall(r"\bT (bsq_\w+)", nm.stdout)))
        assert exported == _declared()


def test_version_and_status_strings(lib):
    assert lib.bsq_version() >> 16 == 1
    for code in range(7):
        assert lib.bsq_status_string(code)
    assert lib.bsq_status_string(99) == b"unknown bsq status"


@pytest.mark.parametrize("fmt,name", [(0, "nvfp4"), (1, "mxfp4"), (2, "mxfp8")])
def test_sizes_match_oracle_layout(lib, fmt, name):
    SF = oracle.block_size(name)
    assert lib.bsq_block_size(fmt) == SF
    for K in (0, 32, 96, 4096, 7168):
        assert lib.bsq_packed_row_bytes(fmt, K) == oracle.packed_row_bytes(name, K)
        for rows in (0, 1, 127, 128, 129, 8192):
            assert lib.bsq_scales5d_bytes(fmt, rows, K) == oracle.scales5d_bytes(rows, K // SF)
    assert lib.bsq_block_size(7) == 0 and lib.bsq_packed_row_bytes(7, 32) == 0
    assert lib.bsq_scales5d_bytes(0, -1, 32) == 0


def q(lib, fmt=0, inp=P, M=128, K=256, ld=256, out=P, sc=P, tsf=1.0):
    return lib.bsq_quantize(fmt, inp, M, K, ld, out, sc, tsf, None)


@pytest.mark.parametrize("kw,code", [
    (dict(fmt=3), VALUE), (dict(fmt=-1), VALUE),
    (dict(M=-1), SHAPE), (dict(K=-32), SHAPE), (dict(K=48, ld=48), SHAPE), (dict(K=16, ld=16), SHAPE),
    (dict(M=1 << 31), SHAPE), (dict(ld=128), SHAPE),
    (dict(inp=None), NULL), (dict(out=None), NULL), (dict(sc=None), NULL),
    (dict(inp=P + 8), ALIGN), (dict(out=P + 4), ALIGN), (dict(sc=P + 1), ALIGN), (dict(ld=260), ALIGN),
    (dict(tsf=0.0), VALUE), (dict(tsf=-1.0), VALUE), (dict(tsf=float("inf")), VALUE),
    (dict(tsf=float("nan")), VALUE),
    (dict(M=0), OK), (dict(K=0, ld=0), OK), (dict(M=0, inp=None, out=None, sc=None), OK),
])
def test_quantize_validation(lib, kw, code):
    assert q(lib, **kw) == code


def test_quantize_mx_ignores_tensor_sf_validation(lib):
    # MX formats ignore tensor_sf, so a bad value does not fail validation; probe with a
    # NULL input so the call still stops before CUDA
    assert q(lib, fmt=1, tsf=float("nan"), inp=None) == NULL
    assert q(lib, fmt=0, tsf=float("nan"), inp=None) == NULL  # NULL is checked first


def g(lib, fmt=0, inp=P, in_rows=64, K=256, ld=256, ro=P, so=P, eid=P, sf=P, ne=8, ridx=None,
      G=4, total_rows=64, total_scale_rows=512, out=P, sc=P, kt=1):
    return lib.bsq_grouped_quantize(fmt, inp, in_rows, K, ld, ro, so, eid, sf, ne, ridx, G,
                                    total_rows, total_scale_rows, out, sc, kt, None)


@pytest.mark.parametrize("kw,code", [
    (dict(fmt=5), VALUE), (dict(kt=3), VALUE), (dict(kt=-1), VALUE), (dict(kt=16), VALUE),
    (dict(kt=0, G=0), OK),
    (dict(G=-1), VALUE), (dict(G=(1 << 20) + 1), VALUE),
    (dict(K=100, ld=100), SHAPE), (dict(in_rows=-1), SHAPE), (dict(total_rows=-1), SHAPE),
    (dict(total_scale_rows=100), SHAPE), (dict(ld=128), SHAPE),
    (dict(inp=None), NULL), (dict(ro=None), NULL), (dict(so=None), NULL), (dict(eid=None), NULL),
    (dict(out=None), NULL), (dict(sc=None), NULL), (dict(sf=None), NULL),
    (dict(ne=0), VALUE),
    (dict(inp=P + 2), ALIGN), (dict(ld=260), ALIGN), (dict(out=P + 8), ALIGN), (dict(sc=P + 4), ALIGN),
    (dict(ro=P + 2), ALIGN), (dict(ridx=P + 1), ALIGN),
    (dict(G=0), OK), (dict(K=0, ld=0), OK), (dict(total_scale_rows=0), OK),
])
def test_grouped_validation(lib, kw, code):
    assert g(lib, **kw) == code


def test_grouped_mx_allows_null_sf(lib):
    # MX formats read no sf: NULL sf passes that check and the call stops at the next one
    assert g(lib, fmt=2, sf=None, ne=0, out=None) == NULL
    assert g(lib, fmt=2, sf=None, ne=0, out=P + 8) == ALIGN


def il(lib, inp=P, M=100, S=20, ld=20, out=P):
    return lib.bsq_scales_interleave(inp, M, S, ld, out, None)


@pytest.mark.parametrize("kw,code", [
    (dict(M=-1), SHAPE), (dict(S=-1), SHAPE), (dict(ld=19), SHAPE),
    (dict(inp=None), NULL), (dict(out=None), NULL), (dict(out=P + 8), ALIGN),
    (dict(M=0), OK), (dict(S=0, ld=0), OK), (dict(M=0, inp=None, out=None), OK),
])
def test_interleave_validation(lib, kw, code):
    assert il(lib, **kw) == code


def test_device_error_rejects_null_out(lib):
    assert lib.bsq_device_error(None, None) == NULL


def test_binding_raises_readable_errors(lib):
    import fp8_activation_quantization_bsq_gb300 as bsq
    err = bsq.BsqError(SHAPE, "bsq_quantize")
    assert "BSQ_ERR_SHAPE" in str(err) and err.code == SHAPE


def test_grouped_kernel_choice_validation(lib):
    lib.bsq_grouped_quantize_kernel.restype = ctypes.c_int32
    lib.bsq_grouped_quantize_kernel.argtypes = [
        ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
        ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]

    def call(kernel, out=P):
        return lib.bsq_grouped_quantize_kernel(0, P, 64, 256, 256, P, P, P, P, 8, None, 4, 64, 512,
                                               out, P, 1, kernel, None)
    assert call(4, out=None) == VALUE and call(-1, out=None) == VALUE
    for k in (0, 1, 2, 3):
        assert call(k, out=None) == NULL      # valid choice: stops at the next check


def test_tensor_scale_validation(lib):
    ws = lib.bsq_tensor_sf_workspace_bytes()
    assert ws >= 16 + 4 * 1024
    f = lib.bsq_tensor_sf
    f.restype = ctypes.c_int32
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    assert f(P, 4, 12, 12, P, P, ws, None) == SHAPE          # K % 8
    assert f(P, -1, 16, 16, P, P, ws, None) == SHAPE
    assert f(P, 4, 16, 8, P, P, ws, None) == SHAPE           # ld < K
    assert f(P, 4, 16, 16, P, P, ws - 1, None) == SHAPE      # workspace too small
    assert f(None, 4, 16, 16, P, P, ws, None) == NULL
    assert f(P, 4, 16, 16, None, P, ws, None) == NULL
    assert f(P, 4, 16, 16, P, None, ws, None) == NULL
    assert f(P + 8, 4, 16, 16, P, P, ws, None) == ALIGN
    assert f(P, 4, 16, 16, P + 2, P, ws, None) == ALIGN
    assert f(P, 4, 16, 16, P, P + 4, ws, None) == ALIGN
    g = lib.bsq_grouped_tensor_sf
    g.restype = ctypes.c_int32
    g.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    gws = lib.bsq_grouped_tensor_sf_workspace_bytes(8)
    assert gws == 16 + 32 and lib.bsq_grouped_tensor_sf_workspace_bytes(0) == 0
    assert g(P, 64, 256, 256, P, P, None, 4, 64, P, 0, P, gws, None) == VALUE
    assert g(P, 64, 256, 256, P, P, None, -1, 64, P, 8, P, gws, None) == VALUE
    assert g(P, 64, 100, 100, P, P, None, 4, 64, P, 8, P, gws, None) == SHAPE
    assert g(P, 64, 256, 256, P, P, None, 4, 64, P, 8, P, gws - 1, None) == SHAPE
    assert g(P, 64, 256, 256, None, P, None, 4, 64, P, 8, P, gws, None) == NULL
    assert g(P, 64, 256, 256, P, P, None, 4, 64, None, 8, P, gws, None) == NULL
    assert g(P, 64, 256, 256, P, P, P + 1, 4, 64, P, 8, P, gws, None) == ALIGN
    q = lib.bsq_quantize_dynamic
    q.restype = ctypes.c_int32
    q.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert q(0, P, 128, 256, 256, P, P, None, None) == NULL      # NVFP4 needs the scale
    assert q(0, P, 128, 256, 256, P, P, P + 2, None) == ALIGN
    assert q(1, P, 128, 48, 48, P, P, None, None) == SHAPE
    assert q(0, P, 0, 256, 256, None, None, None, None) == OK     # empty: no-op


def test_block_scaled_dot_validation(lib):
    f = lib.bsq_block_scaled_dot
    f.restype = ctypes.c_int32
    f.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_float, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_void_p]
    assert f(3, P, P, 1.0, P, P, 1.0, 4, 4, 64, P, None) == VALUE      # format
    assert f(0, P, P, 1.0, P, P, 1.0, 4, 4, 48, P, None) == SHAPE      # K % 32
    assert f(0, P, P, 1.0, P, P, 1.0, -1, 4, 64, P, None) == SHAPE
    assert f(0, P, P, 1.0, P, P, 1.0, 4, 4, 64, None, None) == NULL
    assert f(0, None, P, 1.0, P, P, 1.0, 4, 4, 64, P, None) == NULL
    assert f(0, P, P, 1.0, P, P, 1.0, 4, 4, 64, P + 4, None) == ALIGN
    assert f(0, P, P, 0.0, P, P, 1.0, 4, 4, 64, P, None) == VALUE      # NVFP4 tensor scale
    assert f(0, P, P, 1.0, P, P, 1.0, 0, 4, 64, None, None) == OK      # empty: no-op


def test_gemm_quantize_validation(lib):
    """Every rejected call returns before anything is enqueued (no valid
    call is made with the fake pointer)."""
    f = lib.bsq_gemm_quantize
    f.restype = ctypes.c_int32
    f.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]

    def call(fmt=1, a=P, b=P, M=64, N=128, K=64, lda=64, ldb=64, tsf=1.0, out=P, sc=P, c=None):
        return f(fmt, a, b, M, N, K, lda, ldb, tsf, out, sc, c, None)
    assert call(fmt=3, out=None) == VALUE
    assert call(N=192, out=None) == SHAPE           # N % 128
    assert call(K=48, lda=48, ldb=48, out=None) == SHAPE   # K % 32
    assert call(M=-1, out=None) == SHAPE
    assert call(K=0, lda=0, ldb=0, out=None) == SHAPE
    assert call(lda=32, out=None) == SHAPE          # lda < K
    assert call(a=None) == NULL
    assert call(out=None) == NULL
    assert call(sc=None) == NULL
    assert call(a=P + 2) == ALIGN
    assert call(K=32, lda=36, ldb=32) == ALIGN      # lda % 8
    assert call(c=P + 4) == ALIGN
    assert call(fmt=0, tsf=0.0) == VALUE            # NVFP4 tensor scale
    assert call(fmt=0, tsf=float("inf")) == VALUE
    assert call(M=0, a=None, b=None, out=None, sc=None) == OK   # empty: no-op



def test_grouped_workspace_validation(lib):
    """bsq_grouped_quantize_ws: the workspace size helper, a misaligned
    workspace (BSQ_ERR_ALIGN), a short one (BSQ_ERR_SHAPE), and a NULL one
    (the call goes on to its other checks)."""
    lib.bsq_grouped_quantize_workspace_bytes.restype = ctypes.c_int64
    lib.bsq_grouped_quantize_workspace_bytes.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int64]
    lib.bsq_scales5d_bytes.restype = ctypes.c_int64
    lib.bsq_scales5d_bytes.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int64]
    for fmt in (0, 1, 2):
        for rows, K in ((512, 256), (128, 96), (0, 64), (384, 7168)):
            bands = rows // 128
            assert lib.bsq_grouped_quantize_workspace_bytes(fmt, rows, K) == \
                lib.bsq_scales5d_bytes(fmt, rows, K) + -(-bands * 4 // 16) * 16
    assert lib.bsq_grouped_quantize_workspace_bytes(3, 128, 64) == 0
    assert lib.bsq_grouped_quantize_workspace_bytes(0, -1, 64) == 0
    f = lib.bsq_grouped_quantize_ws
    f.restype = ctypes.c_int32
    f.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_void_p]
    need = lib.bsq_grouped_quantize_workspace_bytes(0, 512, 256)

    def call(ws, ws_bytes, out=P):
        return f(0, P, 64, 256, 256, P, P, P, P, 8, None, 4, 64, 512, out, P, 1, 3, ws, ws_bytes, None)
    assert call(P + 4, need) == ALIGN
    assert call(P, need - 1) == SHAPE
    assert call(None, 0, out=None) == NULL
    assert call(P, need, out=None) == NULL
