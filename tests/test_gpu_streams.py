"""The entry points on several streams at once: the dense quantize on one
stream and the scale reinterleave of other data on a second stream, forked
from the first at every step and joined at the end (the benchmark step's
arrangement), over rotating buffer sets.  Every result must equal the
oracle's bit for bit, so running the two concurrently on shared SMs changes
nothing."""
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


def test_quantize_and_side_stream_interleave(bsq):
    M, K = 2048, 4096
    S = K // 16
    tsf = 0.5
    sets = []
    for seed in range(3):
        bits = wl.dense_activations(np.random.Generator(np.random.PCG64(90 + seed)), M, K, "rowlognormal")
        s2 = np.random.Generator(np.random.PCG64(190 + seed)).integers(0, 256, size=(M, S), dtype=np.uint8)
        sets.append(dict(bits=bits, x=to_device_bf16(bits), s2=torch.from_numpy(s2).cuda(),
                         out=torch.empty((M, K // 2), dtype=torch.uint8, device="cuda"),
                         sc=torch.empty(oracle.scales5d_bytes(M, S), dtype=torch.uint8, device="cuda"),
                         s5=torch.empty(oracle.scales5d_bytes(M, S), dtype=torch.uint8, device="cuda")))
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    fork = torch.cuda.Event()
    for i in range(12):
        st = sets[i % 3]
        fork.record(main)
        side.wait_event(fork)
        bsq.quantize(st["x"], "nvfp4", tsf, out=st["out"], scales=st["sc"])
        with torch.cuda.stream(side):
            bsq.scales_interleave(st["s2"], out=st["s5"])
    main.wait_stream(side)
    torch.cuda.synchronize()
    for st in sets:
        p_ref, s_ref = oracle.quantize("nvfp4", st["bits"], np.float32(tsf))
        np.testing.assert_array_equal(st["out"].cpu().numpy(), p_ref)
        np.testing.assert_array_equal(st["sc"].cpu().numpy(), s_ref)
        s2 = st["s2"].cpu().numpy()
        np.testing.assert_array_equal(st["s5"].cpu().numpy(), oracle.scales_to_5d(s2))
    assert bsq.device_error() == 0
