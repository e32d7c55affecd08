"""The entry points can be captured into a CUDA graph and replayed: dense
quantize + scale reinterleave, the device-side chain tensor_sf ->
quantize_dynamic (its workspace leaves itself zeroed, so replays need no
memset), and the grouped token kernel with and without its scale-staging
workspace.  Each replay runs on new input copied into the captured buffers
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


@pytest.mark.parametrize("ws", [False, True])
def test_graph_grouped_token_quantize(bsq, ws):
    """The grouped quantize through the token kernel (and, with the
    scale-staging workspace, its second kernel) captured once and replayed
    on new token rows: packed rows and written scale bytes equal the
    oracle on every replay."""
    d = wl.config_grouped_prefill(seed=61, tokens=300, K=256, num_experts=16, top_k=4)
    u32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.uint32).view(np.int32)).cuda()
    ro, so = u32(d["row_offsets"]), u32(d["scales_offsets"])
    eid = torch.from_numpy(d["expert_ids"]).cuda()
    sf = torch.from_numpy(d["sf_tensor"]).cuda()
    ridx = torch.from_numpy(d["row_indices"]).cuda()
    x = torch.empty((300, 256), dtype=torch.bfloat16, device="cuda")
    tsr = d["total_scale_rows"]
    w = torch.empty(bsq.grouped_quantize_workspace_bytes("nvfp4", tsr, 256), dtype=torch.uint8,
                    device="cuda") if ws else None
    kw = dict(total_rows=d["total_rows"], total_scale_rows=tsr, k_tiles_per_block=1, kernel="token", workspace=w)
    out, sc = bsq.grouped_quantize(x, "nvfp4", ro, so, eid, sf, ridx, **kw)   # set-up before capture
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        bsq.grouped_quantize(x, "nvfp4", ro, so, eid, sf, ridx, out=out, scales=sc, **kw)
    for seed in (1, 2):
        rng = np.random.Generator(np.random.PCG64(70 + seed))
        bits = wl.dense_activations(rng, 300, 256, "blocklognormal")
        _bits_to_dev(bits, x)
        p_ref, pw, s_ref, sw = oracle.grouped_quantize("nvfp4", bits, d["row_offsets"], d["scales_offsets"],
                                                       d["expert_ids"], d["sf_tensor"], d["row_indices"])
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy()[pw], p_ref[pw])
        np.testing.assert_array_equal(sc.cpu().numpy()[sw], s_ref[sw])
    assert bsq.device_error() == 0


def test_graph_grouped_dynamic_chain(bsq):
    """Per-expert tensor scales (the token-major reduction: a gather that
    reuses source rows) feeding the grouped NVFP4 quantize from device
    memory, captured once and replayed on new token rows: the workspace
    leaves itself zeroed, so every replay computes fresh scales, and scales,
    packed rows and scale bytes equal the oracle."""
    d = wl.config_grouped_prefill(seed=63, tokens=700, K=512, num_experts=24, top_k=8)
    E = 24
    T, K = 700, 512
    u32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.uint32).view(np.int32)).cuda()
    ro, so = u32(d["row_offsets"]), u32(d["scales_offsets"])
    eid = torch.from_numpy(d["expert_ids"]).cuda()
    ridx = torch.from_numpy(d["row_indices"]).cuda()
    x = torch.zeros((T, K), dtype=torch.bfloat16, device="cuda")
    gws = torch.zeros(bsq.lib().bsq_grouped_tensor_sf_workspace_bytes(E), dtype=torch.uint8, device="cuda")
    sf = bsq.grouped_tensor_sf(x, ro, eid, E, ridx, total_rows=d["total_rows"], workspace=gws)
    kw = dict(total_rows=d["total_rows"], total_scale_rows=d["total_scale_rows"])
    out, sc = bsq.grouped_quantize(x, "nvfp4", ro, so, eid, sf, ridx, **kw)   # set-up before capture
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        bsq.grouped_tensor_sf(x, ro, eid, E, ridx, total_rows=d["total_rows"], out=sf, workspace=gws)
        bsq.grouped_quantize(x, "nvfp4", ro, so, eid, sf, ridx, out=out, scales=sc, **kw)
    for seed in (1, 2, 3):
        rng = np.random.Generator(np.random.PCG64(80 + seed))
        bits = wl.dense_activations(rng, T, K, "rowlognormal")
        _bits_to_dev(bits, x)
        _, sf_ref = oracle.expert_tensor_sf(bits, d["row_offsets"], d["expert_ids"], E, d["row_indices"])
        p_ref, pw, s_ref, sw = oracle.grouped_quantize("nvfp4", bits, d["row_offsets"], d["scales_offsets"],
                                                       d["expert_ids"], sf_ref, d["row_indices"])
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(sf.cpu().numpy(), sf_ref)
        np.testing.assert_array_equal(out.cpu().numpy()[pw], p_ref[pw])
        np.testing.assert_array_equal(sc.cpu().numpy()[sw], s_ref[sw])
    assert int(gws.count_nonzero().item()) == 0
    assert bsq.device_error() == 0
