"""Consumer-side check of the quantized operands on the tensor cores.

The packed elements and 5D scales written by the quantize kernels go, as
they are, into torch._scaled_mm (cuBLASLt's block-scaled GEMM, which runs on
the tcgen05 tensor cores and reads the scales in the swizzled 128 x 4 tile
layout), and the product is compared with the oracle's dequantise-then-dot
(float64, scales read through the 5D layout statement).  If the kernels'
nibble order or scale layout differed from what the hardware consumes, the
two would disagree by the size of the product itself, far beyond the FP32
accumulation tolerance used here; a negative control feeds the same scales
in plain row-major order and checks that the disagreement is then gross.

This follows the idea of the naive reference matmul on the
"block_scaled_quantization" module page (function list): check quantized
operands through the layout the tensor cores read.  The library GEMM is only
an independent consumer here, not part of the quantization path.
"""
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


ELEM = {"nvfp4": "float4_e2m1fn_x2", "mxfp4": "float4_e2m1fn_x2", "mxfp8": "float8_e4m3fn"}
SCALE = {"nvfp4": "float8_e4m3fn", "mxfp4": "float8_e8m0fnu", "mxfp8": "float8_e8m0fnu"}


def _operand(bsq, fmt, bits):
    x = to_device_bf16(bits)
    tsf = float(oracle.tensor_sf(bits)[1]) if fmt == "nvfp4" else 1.0
    packed, scales = bsq.quantize(x, fmt, tsf)
    return packed, scales, tsf


def _hw_product(fmt, pa, sa, pb, sb):
    """torch._scaled_mm on the raw bytes; None (with the reason) if this
    torch / GPU does not take block-scaled operands of this format."""
    if not hasattr(torch, ELEM[fmt]) or not hasattr(torch, SCALE[fmt]):
        return None, f"torch has no {ELEM[fmt]} / {SCALE[fmt]}"
    a = pa.view(getattr(torch, ELEM[fmt]))
    b = pb.view(getattr(torch, ELEM[fmt])).t()  # (K', N), column-major
    s_a = sa.view(getattr(torch, SCALE[fmt]))
    s_b = sb.view(getattr(torch, SCALE[fmt]))
    last = None
    for out_dtype in (torch.float32, torch.bfloat16):
        try:
            c = torch._scaled_mm(a, b, scale_a=s_a, scale_b=s_b, out_dtype=out_dtype)
            torch.cuda.synchronize()
            return c.float(), out_dtype
        except (RuntimeError, TypeError, ValueError) as e:
            last = e
    return None, f"torch._scaled_mm refused {fmt} operands: {str(last).splitlines()[0][:200]}"


def _plain_row_major(scales5d, rows, S):
    """The same scale bytes rearranged to plain (rows_padded, S_padded) row-major
    order: the layout the hardware does not read (negative control)."""
    buf = scales5d.cpu().numpy()
    m2 = oracle.scales_from_5d_view(buf, rows, S)
    return torch.from_numpy(np.ascontiguousarray(m2).reshape(-1)).cuda()


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("M,N,K", [(256, 128, 512), (384, 256, 1024)])
def test_tensor_core_product_of_quantized_operands(bsq, fmt, M, N, K):
    rng = np.random.Generator(np.random.PCG64(21 + M + K))
    a_bits = wl.dense_activations(rng, M, K, "rowlognormal")
    b_bits = wl.dense_activations(rng, N, K, "blocklognormal")
    pa, sa, tsf_a = _operand(bsq, fmt, a_bits)
    pb, sb, tsf_b = _operand(bsq, fmt, b_bits)
    c_hw, info = _hw_product(fmt, pa, sa, pb, sb)
    if c_hw is None:
        pytest.skip(info)
    # hardware product of the stored values; NVFP4 elements carry 1/tensor_sf
    c_hw = c_hw.double().cpu().numpy() / (tsf_a * tsf_b)
    pa_h, sa_h, pb_h, sb_h = (t.cpu().numpy() for t in (pa, sa, pb, sb))
    c_ref = oracle.naive_block_scaled_matmul(fmt, pa_h, sa_h, tsf_a, pb_h, sb_h, tsf_b, K)
    S = K // oracle.block_size(fmt)
    a_abs = np.abs(oracle.dequantize(fmt, pa_h, oracle.scales_from_5d_view(sa_h, M, S)[:M, :S], tsf_a))
    b_abs = np.abs(oracle.dequantize(fmt, pb_h, oracle.scales_from_5d_view(sb_h, N, S)[:N, :S], tsf_b))
    mag = a_abs @ b_abs.T  # sum of |terms| per output
    rel = 1e-5 if info == torch.float32 else 8e-3
    err = np.abs(c_hw - c_ref)
    assert np.all(err <= rel * mag + 1e-30), f"max err/mag {np.max(err / (mag + 1e-30)):.3g} ({info})"
    # the GPU naive block-scaled matmul reads the same bytes the same way
    c_val = bsq.block_scaled_dot(fmt, pa, sa, pb, sb, K, tsf_a, tsf_b).cpu().numpy()
    assert np.all(np.abs(c_hw - c_val) <= rel * mag + 1e-30)

    # negative control: scales in plain row-major order are not what the
    # tensor cores read, and the product must then be far off
    c_bad, _ = _hw_product(fmt, pa, _plain_row_major(sa, M, S), pb, _plain_row_major(sb, N, S))
    c_bad = c_bad.double().cpu().numpy() / (tsf_a * tsf_b)
    assert np.max(np.abs(c_bad - c_ref) / (mag + 1e-30)) > 100 * rel
