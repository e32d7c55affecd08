"""Device-side failure path without a fault: a bounded wait that nothing
satisfies gives up after about a second, records BSQ_ERR_TIMEOUT in the
error word, and leaves the context usable (a quantize right after it is
still bit-exact)."""
import time

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


def test_bounded_wait_times_out_and_context_stays_usable(bsq):
    assert bsq.device_error() == 0
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    assert bsq.lib().bsq_selftest_wait_timeout(stream) == 0
    assert bsq.device_error() == 6          # BSQ_ERR_TIMEOUT
    assert 0.5 < time.perf_counter() - t0 < 60
    assert bsq.device_error() == 0          # read-and-clear
    c = wl.config_dense_nvfp4_small()
    x = torch.from_numpy(np.ascontiguousarray(c["x_bits"]).view(np.int16)).view(torch.bfloat16).cuda()
    out, sc = bsq.quantize(x, "nvfp4", c["tensor_sf"])
    p_ref, s_ref = oracle.quantize("nvfp4", c["x_bits"], c["tensor_sf"])
    np.testing.assert_array_equal(out.cpu().numpy(), p_ref)
    np.testing.assert_array_equal(sc.cpu().numpy(), s_ref)
