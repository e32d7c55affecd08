"""The entry points can be captured into a CUDA graph and replayed: dense
quantize + scale reinterleave, and the device-side chain tensor_sf ->
quantize_dynamic (its workspace leaves itself zeroed, so replays need no
memset).  Each replay runs on new input copied into the captured buffers
and must match the oracle bit for bit.  Per-device set-up happens on a
first call made before the capture."""
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


def _bits_to_dev(bits, dst):
    dst.copy_(torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16))


def test_graph_dense_quantize_and_interleave(bsq):
    M, K = 384, 1024
    S = K // 16
    x = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    s2 = torch.empty((M, S), dtype=torch.uint8, device="cuda")
    out = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    sc = torch.empty(oracle.scales5d_bytes(M, S), dtype=torch.uint8, device="cuda")
    s5 = torch.empty_like(sc)
    tsf = 0.75
    bsq.quantize(x, "nvfp4", tsf, out=out, scales=sc)      # per-device set-up before capture
    bsq.scales_interleave(s2, out=s5)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        bsq.quantize(x, "nvfp4", tsf, out=out, scales=sc)
        bsq.scales_interleave(s2, out=s5)
    for seed in (1, 2):
        rng = np.random.Generator(np.random.PCG64(50 + seed))
        bits = wl.dense_activations(rng, M, K, "rowlognormal")
        _bits_to_dev(bits, x)
        p_ref, s_ref = oracle.quantize("nvfp4", bits, tsf)
        _, s2_ref = oracle.quantize_rank2("nvfp4", bits, tsf)
        s2.copy_(torch.from_numpy(s2_ref))
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy(), p_ref)
        np.testing.assert_array_equal(sc.cpu().numpy(), s_ref)
        np.testing.assert_array_equal(s5.cpu().numpy(), s_ref)
    assert bsq.device_error() == 0


def test_graph_tensor_scale_chain(bsq):
    M, K = 256, 512
    x = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(bsq.lib().bsq_tensor_sf_workspace_bytes(), dtype=torch.uint8, device="cuda")
    t = torch.empty(2, dtype=torch.float32, device="cuda")
    out = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    sc = torch.empty(oracle.scales5d_bytes(M, K // 16), dtype=torch.uint8, device="cuda")
    x.zero_()
    bsq.tensor_sf(x, out=t, workspace=ws)
    bsq.quantize_dynamic(x, "nvfp4", t[1:], out=out, scales=sc)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        bsq.tensor_sf(x, out=t, workspace=ws)
        bsq.quantize_dynamic(x, "nvfp4", t[1:], out=out, scales=sc)
    for seed in (3, 4, 5):
        rng = np.random.Generator(np.random.PCG64(60 + seed))
        bits = wl.dense_activations(rng, M, K, "outliers1pct")
        _bits_to_dev(bits, x)
        amax, tsf = oracle.tensor_sf(bits)
        p_ref, s_ref = oracle.quantize("nvfp4", bits, tsf)
        g.replay()
        torch.cuda.synchronize()
        got = t.cpu().numpy()
        assert got[0] == amax and got[1] == tsf
        np.testing.assert_array_equal(out.cpu().numpy(), p_ref)
        np.testing.assert_array_equal(sc.cpu().numpy(), s_ref)
    assert bsq.device_error() == 0
