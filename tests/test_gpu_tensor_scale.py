"""GPU parity of the tensor-scale reductions (global and per-expert amax ->
NVFP4 tensor_sf) and of quantize_dynamic, which reads tensor_sf from device
memory, against the CPU oracle: amax and tensor_sf bit-exact, packed bytes
and scales bit-exact."""
import numpy as np
import pytest

import oracle
import workloads as wl
from bsq_testlib import SENTINEL, guarded, i32_device, margin_intact, to_device_bf16, u32_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def bsq():
    import fp8_activation_quantization_bsq_gb300 as m
    from fp8_activation_quantization_bsq_gb300 import _build
    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def _f32(t):
    return t.cpu().numpy().astype(np.float32)


CASES = {
    "small": lambda: wl.config_dense_nvfp4_small()["x_bits"],
    "large": lambda: wl.config_dense_nvfp4_large()["x_bits"],
    "zeros": lambda: np.zeros((70, 64), np.uint16),
    "neg_zero_and_max": lambda: np.array([[0x8000, 0xFF7F] + [0] * 14], np.uint16),
    "one_row": lambda: wl.dense_activations(np.random.Generator(np.random.PCG64(1)), 1, 8, "normal"),
    "many_rows": lambda: wl.dense_activations(np.random.Generator(np.random.PCG64(2)), 40000, 16, "rowlognormal"),
    "subnormal_max": lambda: np.array([[0x0003, 0x8001] * 8], np.uint16),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_tensor_sf_exact(bsq, case):
    bits = CASES[case]()
    x = to_device_bf16(bits)
    out = bsq.tensor_sf(x)
    amax, tsf = oracle.tensor_sf(bits)
    got = _f32(out)
    assert got[0] == amax
    assert got[1] == tsf or (np.isinf(tsf) and np.isinf(got[1]))
    assert bsq.device_error() == 0


def test_tensor_sf_strided_and_workspace_reuse(bsq):
    rng = np.random.Generator(np.random.PCG64(3))
    bits = wl.dense_activations(rng, 300, 96, "rowlognormal")
    wide = np.zeros((300, 136), np.uint16)
    wide[:, :96] = bits
    wide[:, 96:] = 0x7F00                            # huge values outside the view
    x = to_device_bf16(wide)[:, :96]
    ws = torch.zeros(bsq.lib().bsq_tensor_sf_workspace_bytes(), dtype=torch.uint8, device="cuda")
    for _ in range(3):                               # the workspace is reused as is
        out = bsq.tensor_sf(x, workspace=ws)
        amax, tsf = oracle.tensor_sf(bits)
        assert _f32(out)[0] == amax and _f32(out)[1] == tsf
    empty = torch.empty((0, 32), dtype=torch.bfloat16, device="cuda")
    np.testing.assert_array_equal(_f32(bsq.tensor_sf(empty, workspace=ws)), [0.0, 1.0])


# Two kernels serve grouped_tensor_sf: a gather that reuses source rows over
# few tokens (in_rows <= 8 K, at most 1024 groups) reduces each token once and
# scans row_indices; the rest reduce every destination row.  The cases below
# reach both: "no_gather" and "tall_short_K" take the per-row kernel.
@pytest.mark.parametrize("cfg", ["prefill_small", "decode", "negative_ids", "no_gather", "tall_short_K",
                                 "ragged_tokens", "indices_off_16B"])
def test_grouped_tensor_sf_exact(bsq, cfg):
    ridx_used = True
    if cfg == "decode":
        d = wl.config_grouped_decode(K=2048)
        E = 256
    elif cfg == "tall_short_K":
        d = wl.config_grouped_prefill(seed=6, tokens=1100, K=64, num_experts=16, top_k=3)
        E = 16
    elif cfg == "ragged_tokens":                     # a partial last block of tokens
        d = wl.config_grouped_prefill(seed=8, tokens=37, K=512, num_experts=8, top_k=5)
        E = 8
    else:
        d = wl.config_grouped_prefill(seed=5, tokens=200, K=256, num_experts=32, top_k=4)
        E = 32
    eid = d["expert_ids"].copy()
    if cfg == "negative_ids":
        eid[::4] = -1
    x_bits = d["x_bits"]
    if cfg == "no_gather":                           # destination rows are the rows of x
        ridx_used = False
        x_bits = wl.dense_activations(np.random.Generator(np.random.PCG64(9)), d["total_rows"], d["K"],
                                      "rowlognormal")
    x = to_device_bf16(x_bits)
    ridx = d["row_indices"] if ridx_used else None
    ridx_dev = i32_device(ridx) if ridx_used else None
    if cfg == "indices_off_16B":                     # row_indices 4 bytes past a 16-byte boundary
        ridx_dev = i32_device(np.concatenate([[7], ridx]).astype(np.int32))[1:]
    sf = bsq.grouped_tensor_sf(x, u32_device(d["row_offsets"]), i32_device(eid), E, ridx_dev,
                               total_rows=d["total_rows"])
    amax, ref = oracle.expert_tensor_sf(x_bits, d["row_offsets"], eid, E, ridx)
    np.testing.assert_array_equal(_f32(sf), ref)
    assert bsq.device_error() == 0


@pytest.mark.parametrize("tokens,K", [(200, 256), (1100, 64)])
def test_grouped_tensor_sf_reports_bad_source_rows(bsq, tokens, K):
    """A gathered source row outside x (for an expert that is kept) is
    reported (BSQ_ERR_VALUE) and never read, in either kernel; the same row
    in a group with expert -1 is skipped without an error."""
    d = wl.config_grouped_prefill(seed=10, tokens=tokens, K=K, num_experts=8, top_k=2)
    x = to_device_bf16(d["x_bits"])
    ro, eid = d["row_offsets"], d["expert_ids"].copy()
    g = int(np.argmax(np.diff(ro.astype(np.int64)) > 0))     # a group with rows
    ridx = d["row_indices"].copy()
    ridx[ro[g]] = tokens + 5
    assert bsq.device_error() == 0
    bsq.grouped_tensor_sf(x, u32_device(ro), i32_device(eid), 8, i32_device(ridx), total_rows=d["total_rows"])
    assert bsq.device_error() == 4
    eid[g] = -1
    sf = bsq.grouped_tensor_sf(x, u32_device(ro), i32_device(eid), 8, i32_device(ridx),
                               total_rows=d["total_rows"])
    assert bsq.device_error() == 0
    _, ref = oracle.expert_tensor_sf(d["x_bits"], ro, eid, 8, ridx)
    np.testing.assert_array_equal(_f32(sf), ref)


def test_grouped_tensor_sf_no_groups_gives_ones(bsq):
    x = torch.zeros((4, 32), dtype=torch.bfloat16, device="cuda")
    sf = bsq.grouped_tensor_sf(x, u32_device(np.zeros(1, np.uint32)),
                               i32_device(np.zeros(0, np.int32)), 5, total_rows=0)
    np.testing.assert_array_equal(_f32(sf), np.ones(5, np.float32))


@pytest.mark.parametrize("case", ["small", "large"])
def test_quantize_dynamic_chain_matches_oracle(bsq, case):
    """tensor_sf then quantize_dynamic on one stream, no host round trip."""
    bits = CASES[case]()
    M, K = bits.shape
    x = to_device_bf16(bits)
    packed, scales = bsq.quantize_dynamic(x, "nvfp4")
    _, tsf = oracle.tensor_sf(bits)
    if case == "large":
        rows = np.arange(0, M, 97)
        p_ref, s_ref = oracle.quantize_rank2("nvfp4", bits[rows], tsf)
        np.testing.assert_array_equal(packed.cpu().numpy()[rows], p_ref)
        S = K // 16
        mm, ss = np.meshgrid(rows, np.arange(S), indexing="ij")
        np.testing.assert_array_equal(scales.cpu().numpy()[oracle.offset_5d(mm, ss, -(-S // 4))], s_ref)
    else:
        p_ref, s_ref = oracle.quantize("nvfp4", bits, tsf)
        np.testing.assert_array_equal(packed.cpu().numpy(), p_ref)
        np.testing.assert_array_equal(scales.cpu().numpy(), s_ref)
    assert bsq.device_error() == 0


@pytest.mark.parametrize("bad", [0.0, -1.0, float("nan"), float("inf")])
def test_quantize_dynamic_rejects_bad_device_scale(bsq, bad):
    bits = CASES["small"]()
    x = to_device_bf16(bits)
    M, K = bits.shape
    ofull, out = guarded(M * K // 2)
    sfull, sc = guarded(oracle.scales5d_bytes(M, K // 16))
    tsf = torch.tensor([bad], dtype=torch.float32, device="cuda")
    bsq.quantize_dynamic(x, "nvfp4", tsf, out=out, scales=sc)
    assert bsq.device_error() == 4
    assert np.all(ofull.cpu().numpy() == SENTINEL) and np.all(sfull.cpu().numpy() == SENTINEL)


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp8"])
def test_quantize_dynamic_mx_ignores_scale(bsq, fmt):
    bits = CASES["small"]()
    x = to_device_bf16(bits)
    packed, scales = bsq.quantize_dynamic(x, fmt, None)
    p_ref, s_ref = oracle.quantize(fmt, bits)
    np.testing.assert_array_equal(packed.cpu().numpy(), p_ref)
    np.testing.assert_array_equal(scales.cpu().numpy(), s_ref)


def test_workspaces_left_zeroed_and_unzeroed_ones_reported(bsq):
    """Each call leaves its workspace zeroed for the next one; a workspace
    that was never zeroed is reported (BSQ_ERR_VALUE), not silently used."""
    bits = CASES["small"]()
    x = to_device_bf16(bits)
    ws = torch.zeros(bsq.lib().bsq_tensor_sf_workspace_bytes(), dtype=torch.uint8, device="cuda")
    bsq.tensor_sf(x, workspace=ws)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero().item()) == 0          # counter and running maximum back to zero
    d = wl.config_grouped_prefill(seed=5, tokens=200, K=256, num_experts=32, top_k=4)
    gws = torch.zeros(bsq.lib().bsq_grouped_tensor_sf_workspace_bytes(32), dtype=torch.uint8, device="cuda")
    args = (to_device_bf16(d["x_bits"]), u32_device(d["row_offsets"]), i32_device(d["expert_ids"]), 32,
            i32_device(d["row_indices"]))
    bsq.grouped_tensor_sf(*args, total_rows=d["total_rows"], workspace=gws)
    torch.cuda.synchronize()
    assert int(gws.count_nonzero().item()) == 0
    assert bsq.device_error() == 0
    bad = torch.full_like(ws, 0xFF)
    bsq.tensor_sf(x, workspace=bad)
    assert bsq.device_error() == 4
    gbad = torch.full_like(gws, 0xFF)
    bsq.grouped_tensor_sf(*args, total_rows=d["total_rows"], workspace=gbad)
    assert bsq.device_error() == 4


@pytest.mark.parametrize("kernel", ["stream", "latency"])
def test_grouped_dynamic_chain_matches_oracle(bsq, kernel):
    """Per-expert tensor scales computed on the GPU feed the grouped NVFP4
    quantize directly (device memory, no host round trip)."""
    d = wl.config_grouped_prefill(seed=7, tokens=160, K=512, num_experts=24, top_k=4)
    E = 24
    x = to_device_bf16(d["x_bits"])
    ro, so = u32_device(d["row_offsets"]), u32_device(d["scales_offsets"])
    eid, ridx = i32_device(d["expert_ids"]), i32_device(d["row_indices"])
    sf = bsq.grouped_tensor_sf(x, ro, eid, E, ridx, total_rows=d["total_rows"])
    out, sc = bsq.grouped_quantize(x, "nvfp4", ro, so, eid, sf, ridx, total_rows=d["total_rows"],
                                   total_scale_rows=d["total_scale_rows"], k_tiles_per_block=2,
                                   kernel=kernel)
    _, sf_ref = oracle.expert_tensor_sf(d["x_bits"], d["row_offsets"], d["expert_ids"], E, d["row_indices"])
    p_ref, pw, s_ref, sw = oracle.grouped_quantize("nvfp4", d["x_bits"], d["row_offsets"], d["scales_offsets"],
                                                   d["expert_ids"], sf_ref, d["row_indices"])
    np.testing.assert_array_equal(out.cpu().numpy()[pw], p_ref[pw])
    np.testing.assert_array_equal(sc.cpu().numpy()[sw], s_ref[sw])
    assert bsq.device_error() == 0


@pytest.mark.parametrize("stale", [1, 0x7FFFFFFF])
def test_stale_counter_is_reported(bsq, stale):
    """A completion counter left non-zero is reported (BSQ_ERR_VALUE) for both
    reductions; with a counter at or past the block count nothing is written
    (the output keeps its sentinel), with a small stale counter the launch is
    reported and its output must be discarded."""
    bits = CASES["large"]()[:2048]
    x = to_device_bf16(bits)
    ws = torch.zeros(bsq.lib().bsq_tensor_sf_workspace_bytes(), dtype=torch.uint8, device="cuda")
    ws[:4].view(torch.int32).fill_(stale)
    out = torch.full((2,), -7.0, dtype=torch.float32, device="cuda")
    bsq.tensor_sf(x, out=out, workspace=ws)
    assert bsq.device_error() == 4
    if stale >= 1024:
        np.testing.assert_array_equal(_f32(out), [-7.0, -7.0])
    d = wl.config_grouped_prefill(seed=5, tokens=200, K=256, num_experts=32, top_k=4)
    gws = torch.zeros(bsq.lib().bsq_grouped_tensor_sf_workspace_bytes(32), dtype=torch.uint8, device="cuda")
    gws[:4].view(torch.int32).fill_(stale)
    gout = torch.full((32,), -7.0, dtype=torch.float32, device="cuda")
    bsq.grouped_tensor_sf(to_device_bf16(d["x_bits"]), u32_device(d["row_offsets"]), i32_device(d["expert_ids"]),
                          32, i32_device(d["row_indices"]), total_rows=d["total_rows"], out=gout, workspace=gws)
    assert bsq.device_error() == 4
    if stale >= 1024:
        assert np.all(_f32(gout) == -7.0)


@pytest.mark.parametrize("kernel", ["auto", "token"])
def test_grouped_quantize_dynamic_matches_oracle(bsq, kernel):
    """One call: per-expert scales on the GPU, then the grouped NVFP4
    quantize reading them from device memory."""
    d = wl.config_grouped_prefill(seed=9, tokens=400, K=1024, num_experts=32, top_k=8)
    E = 32
    x = to_device_bf16(d["x_bits"])
    ro, so = u32_device(d["row_offsets"]), u32_device(d["scales_offsets"])
    eid, ridx = i32_device(d["expert_ids"]), i32_device(d["row_indices"])
    out, sc, sf = bsq.grouped_quantize_dynamic(x, ro, so, eid, E, ridx, total_rows=d["total_rows"],
                                               total_scale_rows=d["total_scale_rows"], kernel=kernel)
    _, sf_ref = oracle.expert_tensor_sf(d["x_bits"], d["row_offsets"], d["expert_ids"], E, d["row_indices"])
    p_ref, pw, s_ref, sw = oracle.grouped_quantize("nvfp4", d["x_bits"], d["row_offsets"], d["scales_offsets"],
                                                   d["expert_ids"], sf_ref, d["row_indices"])
    np.testing.assert_array_equal(sf.cpu().numpy(), sf_ref)
    np.testing.assert_array_equal(out.cpu().numpy()[pw], p_ref[pw])
    np.testing.assert_array_equal(sc.cpu().numpy()[sw], s_ref[sw])
    assert bsq.device_error() == 0
