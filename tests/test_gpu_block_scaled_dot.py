"""GPU naive block-scaled matmul (bsq_block_scaled_dot) against the oracle's
dequantise-then-dot.  The operands are the oracle's own quantized bytes and
5D scales, so this checks the validator independently of the quantize
kernels: FP64 on both sides, different summation orders, agreement to 1e-12
of the sum of |terms|."""
import numpy as np
import pytest

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def bsq():
    import fp8_activation_quantization_bsq_gb300 as m
    from fp8_activation_quantization_bsq_gb300 import _build
    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("M,N,K", [(64, 48, 256), (130, 70, 96), (256, 129, 1024)])
def test_block_scaled_dot_matches_oracle(bsq, fmt, M, N, K):
    rng = np.random.Generator(np.random.PCG64(31 + M + N + K))
    a_bits = wl.dense_activations(rng, M, K, "rowlognormal")
    b_bits = wl.dense_activations(rng, N, K, "blocklognormal")
    tsf_a = float(oracle.tensor_sf(a_bits)[1]) if fmt == "nvfp4" else 1.0
    tsf_b = float(oracle.tensor_sf(b_bits)[1]) if fmt == "nvfp4" else 1.0
    pa, sa = oracle.quantize(fmt, a_bits, tsf_a)
    pb, sb = oracle.quantize(fmt, b_bits, tsf_b)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    c = bsq.block_scaled_dot(fmt, dev(pa), dev(sa), dev(pb), dev(sb), K, tsf_a, tsf_b).cpu().numpy()
    ref = oracle.naive_block_scaled_matmul(fmt, pa, sa, tsf_a, pb, sb, tsf_b, K)
    S = K // oracle.block_size(fmt)
    a_abs = np.abs(oracle.dequantize(fmt, pa, oracle.scales_from_5d_view(sa, M, S)[:M, :S], tsf_a))
    b_abs = np.abs(oracle.dequantize(fmt, pb, oracle.scales_from_5d_view(sb, N, S)[:N, :S], tsf_b))
    mag = a_abs @ b_abs.T
    assert np.all(np.abs(c - ref) <= 1e-12 * mag + 1e-300)
    assert bsq.device_error() == 0


def test_block_scaled_dot_validation(bsq):
    x = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(bsq.BsqError, match="BSQ_ERR_SHAPE"):
        bsq.block_scaled_dot("nvfp4", x.view(4, 16), x, x.view(4, 16), x, 48)       # K % 32
    with pytest.raises(bsq.BsqError, match="BSQ_ERR_VALUE"):
        bsq.block_scaled_dot("nvfp4", x.view(4, 16), x, x.view(4, 16), x, 32, 0.0, 1.0)
