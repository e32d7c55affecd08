"""GPU check of the quantize fused into a matmul epilogue (bsq_gemm_quantize):
C = A B^T with BF16 operands and FP32 accumulation, rounded to BF16 and
quantized without being stored.

Two pins, each independent of the kernel: the packed bytes and 5D scales
equal the oracle's quantization of the kernel's own BF16 C (bit for bit, all
scale bytes including the zero padding rows), and that BF16 C equals the
FP64 product within the FP32-accumulation and BF16-rounding bound.  The
fused call without the C copy gives the same bytes."""
import numpy as np
import pytest

import oracle
import workloads as wl
from bsq_testlib import to_device_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def bsq():
    import fp8_activation_quantization_bsq_gb300 as m
    from fp8_activation_quantization_bsq_gb300 import _build
    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def _bf16_to_f64(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("M,N,K,lda_pad", [(128, 128, 64, 0), (200, 256, 96, 8), (1, 128, 32, 0),
                                           (333, 384, 160, 16), (64, 512, 1024, 0)])
def test_fused_epilogue_equals_quantize_of_its_bf16_product(bsq, fmt, M, N, K, lda_pad):
    rng = np.random.Generator(np.random.PCG64(M + N + K))
    a_bits = wl.dense_activations(rng, M, K + lda_pad, "rowlognormal")
    b_bits = wl.dense_activations(rng, N, K, "normal")
    a = to_device_bf16(a_bits)[:, :K]                  # row stride K + lda_pad
    b = to_device_bf16(b_bits)
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    # tensor scale of C from a first pass (delayed scaling), then the checked call
    bsq.gemm_quantize(a, b, fmt, 1.0, c_out=c)
    c_bits = c.view(torch.int16).cpu().numpy().view(np.uint16)
    tsf = float(oracle.tensor_sf(c_bits)[1]) if fmt == "nvfp4" else 1.0
    out, sc = bsq.gemm_quantize(a, b, fmt, tsf, c_out=c)
    c_bits = c.view(torch.int16).cpu().numpy().view(np.uint16)
    assert bsq.device_error() == 0
    # (1) the epilogue is the quantize of the BF16 product
    p_ref, s_ref = oracle.quantize(fmt, c_bits, tsf)
    np.testing.assert_array_equal(out.cpu().numpy(), p_ref)
    np.testing.assert_array_equal(sc.cpu().numpy(), s_ref)
    # (2) the BF16 product against FP64
    a64 = _bf16_to_f64(a_bits[:, :K])
    b64 = _bf16_to_f64(b_bits)
    c64 = a64 @ b64.T
    mag = np.abs(a64) @ np.abs(b64).T
    err = np.abs(_bf16_to_f64(c_bits) - c64)
    assert np.all(err <= 2.0 ** -8 * np.abs(c64) + K * 2.0 ** -23 * mag + 1e-30)
    # (3) the fused call without storing C gives the same bytes
    out2, sc2 = bsq.gemm_quantize(a, b, fmt, tsf)
    assert torch.equal(out2, out) and torch.equal(sc2, sc)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8"])
def test_fused_epilogue_full_size_persistent_tiles(bsq, fmt):
    """The benchmark's shape, 8192 x 2048 x 7168: 512 output tiles over the
    persistent CTAs (several tiles per CTA, both tensor-memory accumulators
    reused, the stage ring wrapping many times).  Every packed byte and
    scale byte equals the oracle's quantization of the kernel's own BF16
    product (in 512-row chunks over a spawned process pool), and sampled
    rows of that product match FP64 within the FP32-accumulation bound."""
    from bsq_testlib import oracle_rank2_chunks
    c_cfg = wl.config_dense_nvfp4_large()
    bits = c_cfg["x_bits"]
    M, K, N = 8192, 7168, 2048
    x = to_device_bf16(bits)
    a, b = x, x[4096:4096 + N]
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    tsf = 2688.0 / 64.0 if fmt == "nvfp4" else 1.0
    out, sc = bsq.gemm_quantize(a, b, fmt, tsf, c_out=c)
    c_bits = c.view(torch.int16).cpu().numpy().view(np.uint16)
    assert bsq.device_error() == 0
    refs = oracle_rank2_chunks(fmt, [(c_bits[r0:r0 + 512], np.float32(tsf)) for r0 in range(0, M, 512)])
    np.testing.assert_array_equal(out.cpu().numpy(), np.concatenate([r[0] for r in refs]))
    np.testing.assert_array_equal(sc.cpu().numpy(), oracle.scales_to_5d(np.concatenate([r[1] for r in refs])))
    rng = np.random.Generator(np.random.PCG64(5))
    rows = np.unique(np.concatenate([[0, 127, 128, M - 1], rng.choice(M, 60, replace=False)]))
    a64 = _bf16_to_f64(bits[rows])
    b64 = _bf16_to_f64(bits[4096:4096 + N])
    c64 = a64 @ b64.T
    mag = np.abs(a64) @ np.abs(b64).T
    err = np.abs(_bf16_to_f64(c_bits[rows]) - c64)
    assert np.all(err <= 2.0 ** -8 * np.abs(c64) + K * 2.0 ** -23 * mag + 1e-30)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("N", [2048, 1920])
def test_fused_epilogue_partial_round_and_tile_column(bsq, fmt, N):
    """2560 x N x 256: 160 output tiles of 128 x 256, more than one round of
    the persistent grid (a partial last round); at N = 1920 the last tile
    column is half outside C.  Bytes equal the oracle's quantize of the
    kernel's own BF16 product, which matches FP64 within the FP32
    accumulation bound."""
    M, K = 2560, 256
    rng = np.random.Generator(np.random.PCG64(N + K))
    a_bits = wl.dense_activations(rng, M, K, "rowlognormal")
    b_bits = wl.dense_activations(rng, N, K, "normal")
    a, b = to_device_bf16(a_bits), to_device_bf16(b_bits)
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    tsf = 3.0 if fmt == "nvfp4" else 1.0
    out, sc = bsq.gemm_quantize(a, b, fmt, tsf, c_out=c)
    c_bits = c.view(torch.int16).cpu().numpy().view(np.uint16)
    assert bsq.device_error() == 0
    p_ref, s_ref = oracle.quantize(fmt, c_bits, np.float32(tsf))
    np.testing.assert_array_equal(out.cpu().numpy(), p_ref)
    np.testing.assert_array_equal(sc.cpu().numpy(), s_ref)
    a64, b64 = _bf16_to_f64(a_bits), _bf16_to_f64(b_bits)
    c64 = a64 @ b64.T
    mag = np.abs(a64) @ np.abs(b64).T
    err = np.abs(_bf16_to_f64(c_bits) - c64)
    assert np.all(err <= 2.0 ** -8 * np.abs(c64) + K * 2.0 ** -23 * mag + 1e-30)
