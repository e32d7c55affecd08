"""The Python binding's own argument checks, on the CPU: they reject what the
C ABI could not describe (wrong dtype, rank, device, stride, names) before
any library call."""
import pytest
import torch

import fp8_activation_quantization_bsq_gb300 as bsq


def test_gemm_quantize_rejects_bad_operands():
    a = torch.zeros((4, 64), dtype=torch.bfloat16)
    b = torch.zeros((128, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        bsq.gemm_quantize(a, b, "nvfp4")                      # host tensors
    with pytest.raises(ValueError):
        bsq.gemm_quantize(a.float(), b, "nvfp4")              # dtype
    with pytest.raises(ValueError):
        bsq.gemm_quantize(a.t(), b, "nvfp4")                  # inner stride


def test_grouped_quantize_rejects_unknown_kernel_and_host_input():
    x = torch.zeros((4, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="kernel"):
        bsq.grouped_quantize(x, "nvfp4", None, None, None, kernel="fastest")
    with pytest.raises(ValueError):
        bsq.grouped_quantize(x, "nvfp4", None, None, None)    # host tensor


def test_quantize_rejects_bad_input_and_format():
    with pytest.raises(ValueError):
        bsq.quantize(torch.zeros((4, 64)), "nvfp4")           # float32
    with pytest.raises(ValueError):
        bsq.quantize(torch.zeros((64,), dtype=torch.bfloat16), "mxfp8")  # rank 1
    with pytest.raises((ValueError, KeyError)):
        bsq.block_size("fp16")


def test_kernel_names_match_the_c_enum():
    assert bsq.GROUPED_KERNELS == {"auto": 0, "stream": 1, "latency": 2, "token": 3}
    text = open(bsq.__file__.replace("fp8_activation_quantization_bsq_gb300/__init__.py", "include/bsq.h")).read()
    for name, value in (("AUTO", 0), ("STREAM", 1), ("LATENCY", 2), ("TOKEN", 3)):
        assert f"BSQ_GROUPED_{name} = {value}" in text
