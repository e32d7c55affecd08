"""GPU parity of the grouped per-expert quantize against the CPU oracle, through
the C ABI (Python binding): bit-exact packed rows and written scale bytes,
sentinel canaries on everything the kernel must leave untouched (rows of
skipped groups, padding scale rows, buffer margins), k_tiles_per_block in
{1, 2, 4, 8}, with and without the row_indices gather, and device-side
bounds checks that turn inconsistent metadata into BSQ_ERR_VALUE.

Operation: grouped_quantize_dynamic_scaled_fp4_async_kernel (Modular
block_scaled_quantization pages).
"""
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


def _run_grouped(bsq, fmt, d, kt, use_ridx=True, expert_ids=None, x_bits=None, ridx=None,
                 expect_error=0, kernel="auto", workspace=False):
    x_bits = d["x_bits"] if x_bits is None else x_bits
    K = x_bits.shape[1]
    eid = d["expert_ids"] if expert_ids is None else expert_ids
    ridx = (d["row_indices"] if use_ridx else None) if ridx is None else ridx
    total_rows, tsr = d["total_rows"], d["total_scale_rows"]
    ob = total_rows * oracle.packed_row_bytes(fmt, K)
    sb = oracle.scales5d_bytes(tsr, K // oracle.block_size(fmt))
    ofull, out = guarded(ob)
    sfull, sc = guarded(sb)
    ws = None
    if workspace:  # staged scale rows; its prior contents must not matter
        wfull, ws = guarded(bsq.grouped_quantize_workspace_bytes(fmt, tsr, K))
        ws.fill_(0xA5)
    bsq.grouped_quantize(to_device_bf16(x_bits), fmt, u32_device(d["row_offsets"]),
                         u32_device(d["scales_offsets"]), i32_device(eid),
                         torch.from_numpy(d["sf_tensor"]).cuda() if fmt == "nvfp4" else None,
                         i32_device(ridx) if ridx is not None else None,
                         total_rows=total_rows, total_scale_rows=tsr, k_tiles_per_block=kt,
                         out=out, scales=sc, kernel=kernel, workspace=ws)
    if workspace:
        assert margin_intact(wfull)
    assert bsq.device_error() == expect_error
    assert margin_intact(ofull) and margin_intact(sfull)
    return out.cpu().numpy().reshape(total_rows, -1), sc.cpu().numpy()


def _compare(fmt, d, p, s, use_ridx=True, expert_ids=None, x_bits=None, ridx=None):
    x_bits = d["x_bits"] if x_bits is None else x_bits
    eid = d["expert_ids"] if expert_ids is None else expert_ids
    ridx = (d["row_indices"] if use_ridx else None) if ridx is None else ridx
    p_ref, pw, s_ref, sw = oracle.grouped_quantize(fmt, x_bits, d["row_offsets"],
                                                   d["scales_offsets"], eid, d["sf_tensor"], ridx)
    np.testing.assert_array_equal(p[pw], p_ref[pw])
    np.testing.assert_array_equal(s[sw], s_ref[sw])
    assert np.all(p[~pw] == SENTINEL), "rows of skipped groups were written"
    assert np.all(s[~sw] == SENTINEL), "padding scale rows were written"


KERNELS = ["stream", "latency", "token"]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("kt", [1, 2, 4, 8])
@pytest.mark.parametrize("K", [256, 96, 1120])
def test_grouped_small(bsq, fmt, kt, K, kernel):
    d = wl.config_grouped_prefill(seed=K + kt, tokens=96, K=K, num_experts=16, top_k=4, fmt=fmt)
    p, s = _run_grouped(bsq, fmt, d, kt, kernel=kernel)
    _compare(fmt, d, p, s)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
def test_grouped_exhaustive_amax_per_expert(bsq, fmt, kernel):
    """Every BF16 block amax through the grouped kernels, with a different
    tensor_sf per expert (NVFP4): scale bytes and codes bit-exact."""
    from test_gpu_dense import _amax_sweep_matrix
    SF = oracle.block_size(fmt)
    mat = _amax_sweep_matrix(SF, per_row_blocks=16)             # 2040 rows x 16 blocks
    rows = mat.shape[0]
    G = 24
    rng = np.random.Generator(np.random.PCG64(77))
    cuts = np.sort(rng.choice(np.arange(1, rows), G - 1, replace=False))
    m = np.diff(np.concatenate([[0], cuts, [rows]]))
    ro = np.concatenate([[0], np.cumsum(m)]).astype(np.uint32)
    so = np.concatenate([[0], np.cumsum((m + 127) // 128 * 128)]).astype(np.uint32)
    sf = np.array([1.0, 0.6640316, 1e-20, 1e20, 2688.0, 3.0e-3] * 8, np.float32)[:G]
    d = dict(x_bits=mat, row_offsets=ro, scales_offsets=so, expert_ids=np.arange(G, dtype=np.int32),
             sf_tensor=sf, row_indices=rng.permutation(rows).astype(np.int32),
             total_rows=rows, total_scale_rows=int(so[-1]), G=G)
    for kt in (1, 4):
        p, s = _run_grouped(bsq, fmt, d, kt, kernel=kernel)
        _compare(fmt, d, p, s)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8"])
def test_grouped_identity_rows(bsq, fmt, kernel):
    d = wl.config_grouped_prefill(seed=1, tokens=64, K=512, num_experts=8, top_k=2, fmt=fmt)
    # without row_indices the destination row d reads source row d
    x = wl.dense_activations(np.random.Generator(np.random.PCG64(2)), d["total_rows"], 512, "blocklognormal")
    p, s = _run_grouped(bsq, fmt, d, 2, use_ridx=False, x_bits=x, kernel=kernel)
    _compare(fmt, d, p, s, use_ridx=False, x_bits=x)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_grouped_large_groups_span_tiles(bsq, fmt, kernel):
    # few experts, many rows each: groups span several 128-row tiles
    d = wl.config_grouped_prefill(seed=9, tokens=600, K=320, num_experts=4, top_k=2, fmt=fmt)
    assert max(np.diff(d["row_offsets"])) > 256
    p, s = _run_grouped(bsq, fmt, d, 4, kernel=kernel)
    _compare(fmt, d, p, s)


@pytest.mark.parametrize("kernel", KERNELS)
def test_grouped_negative_expert_ids_are_skipped(bsq, kernel):
    d = wl.config_grouped_prefill(seed=4, tokens=80, K=256, num_experts=16, top_k=4)
    eid = d["expert_ids"].copy()
    eid[::3] = -1
    p, s = _run_grouped(bsq, "nvfp4", d, 1, expert_ids=eid, kernel=kernel)
    _compare("nvfp4", d, p, s, expert_ids=eid)


def test_grouped_many_groups_search(bsq):
    """G = 3000 one- to three-row groups: more than two rounds of the
    warp-parallel search over scales_offsets."""
    rng = np.random.Generator(np.random.PCG64(6))
    G = 3000
    m = rng.integers(1, 4, size=G)
    ro = np.concatenate([[0], np.cumsum(m)]).astype(np.uint32)
    so = (np.arange(G + 1) * 128).astype(np.uint32)
    x = wl.dense_activations(rng, int(ro[-1]), 64, "blocklognormal")
    d = dict(x_bits=x, row_offsets=ro, scales_offsets=so, expert_ids=np.arange(G, dtype=np.int32),
             sf_tensor=np.ones(G, np.float32), row_indices=rng.permutation(int(ro[-1])).astype(np.int32),
             total_rows=int(ro[-1]), total_scale_rows=int(so[-1]), G=G)
    for fmt in ("mxfp8", "nvfp4"):
        for kernel in KERNELS:
            p, s = _run_grouped(bsq, fmt, d, 1, kernel=kernel)
            _compare(fmt, d, p, s)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8"])
@pytest.mark.parametrize("K", [7168, 2048])
@pytest.mark.parametrize("kt", [0, 1, 2, 4, 8])
@pytest.mark.parametrize("kernel", ["auto", "stream"])
def test_grouped_decode_full_config(bsq, fmt, K, kt, kernel):
    """Decode: 64 tokens, top-8 over 256 experts (512 rows, many 1-row
    experts), row_indices gather -- fully compared (kt = 0: the library
    chooses k_tiles_per_block)."""
    d = wl.config_grouped_decode(K=K, fmt=fmt)
    assert d["total_rows"] / d["G"] <= 8
    p, s = _run_grouped(bsq, fmt, d, kt, kernel=kernel)
    _compare(fmt, d, p, s)


_PREFILL = {}


def _prefill_reference(fmt):
    """The prefill workload (4096 tokens, top-8 of 256 experts, K = 7168:
    32768 destination rows) and the oracle's quantization of every group,
    in row chunks over a spawned process pool; computed once per format."""
    if fmt not in _PREFILL:
        from bsq_testlib import oracle_rank2_chunks
        d = _PREFILL.get("workload")
        if d is None:
            d = _PREFILL["workload"] = wl.config_grouped_prefill()
        ro, eid = d["row_offsets"].astype(np.int64), d["expert_ids"]
        chunks, jobs = [], []
        for gi in range(d["G"]):
            tsf = np.float32(d["sf_tensor"][eid[gi]]) if fmt == "nvfp4" else np.float32(1.0)
            for r0 in range(int(ro[gi]), int(ro[gi + 1]), 512):
                r1 = min(r0 + 512, int(ro[gi + 1]))
                chunks.append((gi, r0, r1))
                jobs.append((d["x_bits"][d["row_indices"][r0:r1]], tsf))
        _PREFILL[fmt] = (chunks, oracle_rank2_chunks(fmt, jobs))
    return _PREFILL["workload"], _PREFILL[fmt]


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8", "mxfp4"])
@pytest.mark.parametrize("kernel", ["auto", "token", "stream", "token+workspace", "auto+workspace"])
def test_grouped_prefill_full_config_all_rows(bsq, fmt, kernel):
    """Prefill at full size (32768 rows, K = 7168) in the benchmark's launch
    configuration (also with the scale-staging workspace): every packed row
    and every written scale byte against the oracle, and the padding scale
    rows (never written) keep their sentinel."""
    d, (chunks, refs) = _prefill_reference(fmt)
    p, s = _run_grouped(bsq, fmt, d, 8, kernel=kernel.split("+")[0], workspace=kernel.endswith("+workspace"))
    K = d["K"]
    S = K // oracle.block_size(fmt)
    Kt = -(-S // 4)
    written = np.zeros(s.size, bool)
    so, ro = d["scales_offsets"].astype(np.int64), d["row_offsets"].astype(np.int64)
    for (gi, r0, r1), (pd, sd) in zip(chunks, refs):
        np.testing.assert_array_equal(p[r0:r1], pd, err_msg=f"group {gi} rows {r0}:{r1}")
        full = np.zeros((r1 - r0, Kt * 4), np.uint8)
        full[:, :S] = sd
        srow = so[gi] + (np.arange(r0, r1) - ro[gi])
        mm, ss = np.meshgrid(srow, np.arange(Kt * 4), indexing="ij")
        off = oracle.offset_5d(mm, ss, Kt)
        np.testing.assert_array_equal(s[off], full, err_msg=f"group {gi} scales rows {r0}:{r1}")
        written[off] = True
    assert np.all(s[~written] == SENTINEL), "padding scale rows were written"


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("kernel", ["token", "stream", "latency", "token+workspace"])
def test_grouped_source_row_past_a_full_bucket_offset_indices(bsq, fmt, kernel):
    """row_indices starting 4 bytes past a 16-byte boundary (a scalar head of
    three entries), a row count that is not a multiple of 4 (a scalar tail),
    one source row in 40 positions (among them the first three and the last
    three), one in exactly 16 (a full bucket of the token kernel) and one in
    17 (one past it): the token kernel's re-scan path and every part of its
    staged scan, against the oracle."""
    d = wl.config_grouped_prefill(seed=21, tokens=67, K=256, num_experts=8, top_k=3, fmt=fmt)
    assert d["total_rows"] % 4 != 0
    rng = np.random.Generator(np.random.PCG64(22))
    ridx = d["row_indices"].copy()
    ridx[np.isin(ridx, [7, 11, 13])] = 5
    n = ridx.size
    pos = rng.permutation(np.arange(3, n - 3))
    heavy = np.concatenate([[0, 1, 2, n - 3, n - 2, n - 1], pos[:34]])
    ridx[heavy] = 7
    ridx[pos[34:50]] = 11
    ridx[pos[50:67]] = 13
    assert np.sum(ridx == 7) == 40 and np.sum(ridx == 11) == 16 and np.sum(ridx == 13) == 17
    dev = i32_device(np.concatenate([[0, 0, 0, 0, 7], ridx]))[5:]   # 20 bytes into a 16-byte aligned buffer
    assert dev.data_ptr() % 16 == 4
    x_bits = d["x_bits"]
    total_rows, tsr = d["total_rows"], d["total_scale_rows"]
    ob = total_rows * oracle.packed_row_bytes(fmt, 256)
    sb = oracle.scales5d_bytes(tsr, 256 // oracle.block_size(fmt))
    ofull, out = guarded(ob)
    sfull, sc = guarded(sb)
    ws = None
    if kernel.endswith("+workspace"):
        ws = torch.full((bsq.grouped_quantize_workspace_bytes(fmt, tsr, 256),), 0x3C, dtype=torch.uint8, device="cuda")
    bsq.grouped_quantize(to_device_bf16(x_bits), fmt, u32_device(d["row_offsets"]), u32_device(d["scales_offsets"]),
                         i32_device(d["expert_ids"]), torch.from_numpy(d["sf_tensor"]).cuda() if fmt == "nvfp4" else None,
                         dev, total_rows=total_rows, total_scale_rows=tsr, k_tiles_per_block=2, out=out, scales=sc,
                         kernel=kernel.split("+")[0], workspace=ws)
    assert bsq.device_error() == 0
    assert margin_intact(ofull) and margin_intact(sfull)
    _compare(fmt, d, out.cpu().numpy().reshape(total_rows, -1), sc.cpu().numpy(), ridx=ridx)


@pytest.mark.parametrize("kernel", KERNELS)
def test_grouped_bad_row_index_is_reported_not_faulted(bsq, kernel):
    d = wl.config_grouped_prefill(seed=8, tokens=40, K=128, num_experts=8, top_k=2)
    ridx = d["row_indices"].copy()
    bad = [3, len(ridx) - 1]
    ridx[bad[0]] = 10_000_000
    ridx[bad[1]] = -5
    p, s = _run_grouped(bsq, "nvfp4", d, 1, ridx=ridx, expect_error=4, kernel=kernel)
    p_ref, pw, _, _ = oracle.grouped_quantize("nvfp4", d["x_bits"], d["row_offsets"],
                                              d["scales_offsets"], d["expert_ids"],
                                              d["sf_tensor"], np.where(ridx < 0, 0, np.minimum(ridx, 39)))
    good = np.ones(d["total_rows"], bool)
    good[bad] = False
    np.testing.assert_array_equal(p[good], p_ref[good])
    assert np.all(p[bad] == SENTINEL)
    # the error word is cleared by the read
    assert bsq.device_error() == 0


@pytest.mark.parametrize("kernel", KERNELS)
def test_grouped_offsets_beyond_buffers_are_reported(bsq, kernel):
    """row_offsets[G] beyond total_rows: the overflowing group is skipped,
    the error word says BSQ_ERR_VALUE and nothing lands past the buffers."""
    d = wl.config_grouped_prefill(seed=8, tokens=40, K=128, num_experts=8, top_k=2)
    d2 = dict(d)
    d2["total_rows"] = d["total_rows"] - 1
    p, s = _run_grouped(bsq, "nvfp4", d2, 1, expect_error=4, kernel=kernel)
    last = d["G"] - 1
    r0 = int(d["row_offsets"][last])
    p_ref, _, _, _ = oracle.grouped_quantize("nvfp4", d["x_bits"], d["row_offsets"],
                                             d["scales_offsets"], d["expert_ids"],
                                             d["sf_tensor"], d["row_indices"])
    np.testing.assert_array_equal(p[:r0], p_ref[:r0])
    assert np.all(p[r0:] == SENTINEL)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("K", [256, 96])
@pytest.mark.parametrize("kernel", KERNELS)
def test_grouped_source_rows_with_many_copies(bsq, fmt, K, kernel):
    """Source rows gathered into many destination rows: 40 and 17 copies of
    two rows among ordinary top-2 routing, each copy quantized with its own
    group's expert scale."""
    d = wl.config_grouped_prefill(seed=9, tokens=70, K=K, num_experts=24, top_k=2)
    ridx = d["row_indices"].copy()
    rng = np.random.Generator(np.random.PCG64(9))
    pos = rng.permutation(len(ridx))
    ridx[pos[:40]] = 5
    ridx[pos[40:57]] = 37
    d = dict(d, row_indices=ridx)
    p, s = _run_grouped(bsq, fmt, d, 1, kernel=kernel)
    _compare(fmt, d, p, s)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("kernel", KERNELS)
def test_grouped_strided_input_and_16_byte_aligned_outputs(bsq, fmt, kernel):
    """The 16-byte load and store paths: input rows with a stride of K + 8
    elements (not a multiple of 32 bytes) and packed / scale outputs that
    start 16 bytes past a 32-byte boundary."""
    d = wl.config_grouped_prefill(seed=10, tokens=90, K=288, num_experts=12, top_k=3)
    K = d["K"]
    wide = np.zeros((d["x_bits"].shape[0], K + 8), np.uint16)
    wide[:, :K] = d["x_bits"]
    wide[:, K:] = 0x7F00                          # huge values outside the view
    x = to_device_bf16(wide)[:, :K]
    total_rows, tsr = d["total_rows"], d["total_scale_rows"]
    ob = total_rows * oracle.packed_row_bytes(fmt, K)
    sb = oracle.scales5d_bytes(tsr, K // oracle.block_size(fmt))
    ofull, _ = guarded(ob + 16)
    sfull, _ = guarded(sb + 16)
    out, sc = ofull[16:16 + ob], sfull[16:16 + sb]
    assert out.data_ptr() % 32 == 16 and sc.data_ptr() % 32 == 16
    bsq.grouped_quantize(x, fmt, u32_device(d["row_offsets"]), u32_device(d["scales_offsets"]),
                         i32_device(d["expert_ids"]),
                         torch.from_numpy(d["sf_tensor"]).cuda() if fmt == "nvfp4" else None,
                         i32_device(d["row_indices"]), total_rows=total_rows, total_scale_rows=tsr,
                         k_tiles_per_block=2, out=out, scales=sc, kernel=kernel)
    assert bsq.device_error() == 0
    assert margin_intact(ofull) and margin_intact(sfull)
    assert np.all(ofull[:16].cpu().numpy() == SENTINEL) and np.all(sfull[:16].cpu().numpy() == SENTINEL)
    _compare(fmt, d, out.cpu().numpy().reshape(total_rows, -1), sc.cpu().numpy())


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("kernel", KERNELS)
def test_grouped_empty_groups_and_trailing_rows(bsq, fmt, kernel):
    """Groups with no rows between non-empty ones (row_offsets and
    scales_offsets do not advance), a group of 129 rows (two scale tiles),
    and destination rows beyond row_offsets[G], which no group owns and which
    stay untouched."""
    rng = np.random.Generator(np.random.PCG64(13))
    m = np.array([0, 5, 0, 0, 129, 1, 0, 40, 0], np.int64)
    G = m.size
    ro = np.concatenate([[0], np.cumsum(m)]).astype(np.uint32)
    so = np.concatenate([[0], np.cumsum(-(-m // 128) * 128)]).astype(np.uint32)
    total_rows = int(ro[-1]) + 7                     # 7 trailing rows outside every group
    K = 192
    in_rows = 90
    x = wl.dense_activations(rng, in_rows, K, "blocklognormal")
    ridx = rng.integers(0, in_rows, size=total_rows).astype(np.int32)
    eid = np.arange(G, dtype=np.int32) % 5
    sf = (rng.random(5).astype(np.float32) + np.float32(0.5))
    d = dict(x_bits=x, row_offsets=ro, scales_offsets=so, expert_ids=eid, sf_tensor=sf,
             row_indices=ridx, total_rows=total_rows, total_scale_rows=int(so[-1]), G=G)
    p, s = _run_grouped(bsq, fmt, d, 2, kernel=kernel)
    owned = int(ro[-1])
    _compare(fmt, d, p[:owned], s)
    assert np.all(p[owned:] == SENTINEL)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("offset", [0, 1, 3])
def test_grouped_token_split_scan_head_and_tail(bsq, fmt, offset):
    """The token-major kernel's scan of row_indices, split between the blocks
    of each cluster: 701 tokens (six clusters of source rows), 2103
    destination rows (not a multiple of 4) and row_indices starting 0, 4 or
    12 bytes past a 16-byte boundary (the scalar head and tail around the
    16-byte body); then two bad source rows, reported once and left
    unwritten, with every other row still exact."""
    d = wl.config_grouped_prefill(seed=20 + offset, tokens=701, K=192, num_experts=20, top_k=3, fmt=fmt)
    K, total_rows, tsr = d["K"], d["total_rows"], d["total_scale_rows"]
    assert total_rows % 4 != 0
    sf = torch.from_numpy(d["sf_tensor"]).cuda() if fmt == "nvfp4" else None
    for bad in (False, True):
        ridx = d["row_indices"].copy()
        if bad:
            ridx[5], ridx[total_rows - 1] = 701, -3
        padded = i32_device(np.concatenate([np.full(offset, 7, np.int32), ridx]))
        rdev = padded[offset:]
        assert rdev.data_ptr() % 16 == 4 * offset
        ofull, out = guarded(total_rows * oracle.packed_row_bytes(fmt, K))
        sfull, sc = guarded(oracle.scales5d_bytes(tsr, K // oracle.block_size(fmt)))
        bsq.grouped_quantize(to_device_bf16(d["x_bits"]), fmt, u32_device(d["row_offsets"]),
                             u32_device(d["scales_offsets"]), i32_device(d["expert_ids"]), sf, rdev,
                             total_rows=total_rows, total_scale_rows=tsr, k_tiles_per_block=1,
                             out=out, scales=sc, kernel="token")
        assert bsq.device_error() == (4 if bad else 0)
        assert margin_intact(ofull) and margin_intact(sfull)
        p = out.cpu().numpy().reshape(total_rows, -1)
        ok = np.ones(total_rows, bool)
        if bad:
            ok[[5, total_rows - 1]] = False
            assert np.all(p[~ok] == SENTINEL)
        p_ref, pw, s_ref, sw = oracle.grouped_quantize(fmt, d["x_bits"], d["row_offsets"], d["scales_offsets"],
                                                       d["expert_ids"], d["sf_tensor"], d["row_indices"])
        np.testing.assert_array_equal(p[pw & ok], p_ref[pw & ok])
        if not bad:
            np.testing.assert_array_equal(sc.cpu().numpy()[sw], s_ref[sw])


@pytest.mark.parametrize("kernel", KERNELS)
def test_grouped_nvfp4_extreme_tensor_scales(bsq, kernel):
    """NVFP4 tensor scales at and beyond the range where the token kernel's
    per-row factor table is exact (2^-117 .. 2^118; outside it the kernel
    divides): tiny, huge and boundary values, one per expert, every kernel
    bit-exact against the oracle."""
    d = wl.config_grouped_prefill(seed=31, tokens=150, K=256, num_experts=10, top_k=3)
    sf = np.array([1e-37, 2.0 ** -117, 2.0 ** -118, 3e36, 2.0 ** 118, 2.0 ** 119, 6e-36, 1.0, 1e-44, 3.4e38],
                  np.float32)
    d = dict(d, sf_tensor=sf[:10])
    p, s = _run_grouped(bsq, "nvfp4", d, 2, kernel=kernel)
    _compare("nvfp4", d, p, s)


@pytest.mark.parametrize("G", [1024, 1025])
@pytest.mark.parametrize("ws", [False, True])
def test_grouped_token_kernel_group_limit(bsq, G, ws):
    """The token kernel keeps the group metadata of up to 1024 groups in
    shared memory; at 1025 the explicit choice falls back to the band kernel
    (which ignores a workspace).  One- to three-row groups gathered from 900
    tokens (rows reused), with and without the scale-staging workspace."""
    rng = np.random.Generator(np.random.PCG64(G))
    m = rng.integers(1, 4, size=G)
    ro = np.concatenate([[0], np.cumsum(m)]).astype(np.uint32)
    so = (np.arange(G + 1) * 128).astype(np.uint32)
    rows = int(ro[-1])
    x = wl.dense_activations(rng, 900, 128, "blocklognormal")
    d = dict(x_bits=x, row_offsets=ro, scales_offsets=so, expert_ids=np.arange(G, dtype=np.int32),
             sf_tensor=np.linspace(0.5, 2.0, G).astype(np.float32),
             row_indices=rng.integers(0, 900, size=rows).astype(np.int32),
             total_rows=rows, total_scale_rows=int(so[-1]), G=G)
    for fmt in ("nvfp4", "mxfp4"):
        p, s = _run_grouped(bsq, fmt, d, 1, kernel="token", workspace=ws)
        _compare(fmt, d, p, s)



@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("tokens,K,top_k,experts", [(1, 32, 1, 1), (5, 64, 3, 4), (300, 32, 2, 8),
                                                     (77825, 32, 2, 64)])
def test_token_kernel_shapes(bsq, fmt, tokens, K, top_k, experts):
    """The token kernel's edge shapes: one token, K = 32 (a partial atom and
    a single step), more SMs than tokens, and 77825 tokens (more than 512
    per block on 152 SMs, so the grid grows past one block per SM)."""
    d = wl.config_grouped_prefill(seed=tokens + K, tokens=tokens, K=K, num_experts=experts, top_k=top_k, fmt=fmt)
    p, s = _run_grouped(bsq, fmt, d, 1, kernel="token")
    _compare(fmt, d, p, s)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("K", [96, 2112, 7168])
@pytest.mark.parametrize("gather", [True, False])
@pytest.mark.parametrize("ws", [False, True])
def test_token_kernel_band_shapes(bsq, fmt, K, gather, ws):
    """The token kernel on scale bands of every fill: groups of 128, 127,
    129, 256 and 1 rows (whole, partly filled and single-row bands), an empty
    group, a skipped group that spans whole bands, and a group with a
    reserved, unused padding tile; with and without the row_indices gather.
    Every written byte equals the oracle and every padding scale row keeps
    its sentinel.  K = 96 / 2112 / 7168 give 1, 33 and 112 (NVFP4) atoms per
    band row.  With the workspace, the staged scale rows reach exactly the
    same 5D bytes and nothing else."""
    rng = np.random.Generator(np.random.PCG64(K + 7 * gather))
    m = np.array([128, 0, 127, 129, 256, 300, 128, 1], np.int64)
    tiles = -(-m // 128)
    tiles[6] += 1                                   # a reserved, unused tile
    G = m.size
    ro = np.concatenate([[0], np.cumsum(m)]).astype(np.uint32)
    so = np.concatenate([[0], np.cumsum(tiles * 128)]).astype(np.uint32)
    total_rows = int(ro[-1])
    in_rows = 300 if gather else total_rows
    x = wl.dense_activations(rng, in_rows, K, "blocklognormal")
    ridx = rng.integers(0, in_rows, size=total_rows).astype(np.int32) if gather else None
    eid = np.array([0, 1, 2, 3, 4, -1, 5, 6], np.int32)
    sf = (rng.random(7).astype(np.float32) + np.float32(0.5)) * np.float32(100.0)
    d = dict(x_bits=x, row_offsets=ro, scales_offsets=so, expert_ids=eid, sf_tensor=sf,
             row_indices=ridx, total_rows=total_rows, total_scale_rows=int(so[-1]), G=G)
    p, s = _run_grouped(bsq, fmt, d, 8, use_ridx=gather, kernel="token", workspace=ws)
    _compare(fmt, d, p, s, use_ridx=gather)


def test_token_kernel_wide_rows(bsq):
    """The token kernel at K = 32768 (NVFP4: 2048 scale blocks, 512 atoms per
    band row; 64 steps per destination row): a whole band and a 5-row band,
    bytes equal to the oracle."""
    rng = np.random.Generator(np.random.PCG64(31))
    m = np.array([128, 5], np.int64)
    ro = np.concatenate([[0], np.cumsum(m)]).astype(np.uint32)
    so = np.concatenate([[0], np.cumsum(-(-m // 128) * 128)]).astype(np.uint32)
    K, in_rows = 32768, 40
    x = wl.dense_activations(rng, in_rows, K, "normal")
    ridx = rng.integers(0, in_rows, size=int(ro[-1])).astype(np.int32)
    d = dict(x_bits=x, row_offsets=ro, scales_offsets=so, expert_ids=np.array([1, 0], np.int32),
             sf_tensor=np.array([3.0, 0.25], np.float32), row_indices=ridx, total_rows=int(ro[-1]),
             total_scale_rows=int(so[-1]), G=2)
    p, s = _run_grouped(bsq, "nvfp4", d, 8, kernel="token")
    _compare("nvfp4", d, p, s)


@pytest.mark.parametrize("n_bad", [2, 100])
@pytest.mark.parametrize("skipped", [False, True])
def test_token_kernel_bad_source_rows_list_and_rescan(bsq, n_bad, skipped):
    """Source rows outside x seen by the token kernel's scan: a few (kept in
    its list and checked once the metadata is in shared memory) and 100
    (more than the list holds: checked by a second pass over row_indices).
    In a kept group they are reported (BSQ_ERR_VALUE) and their rows left
    untouched; in a skipped group (negative expert id) nothing is reported.
    Every other row equals the oracle."""
    d = wl.config_grouped_prefill(seed=17, tokens=600, K=64, num_experts=8, top_k=2)
    g = int(np.argmax(np.diff(d["row_offsets"].astype(np.int64))))      # the largest group
    r0, r1 = int(d["row_offsets"][g]), int(d["row_offsets"][g + 1])
    assert r1 - r0 >= n_bad
    rng = np.random.Generator(np.random.PCG64(n_bad))
    bad = np.sort(rng.choice(np.arange(r0, r1), n_bad, replace=False))
    ridx = d["row_indices"].copy()
    ridx[bad] = np.where(np.arange(n_bad) % 2 == 0, -3, 600 + np.arange(n_bad))
    eid = d["expert_ids"].copy()
    if skipped:
        eid[g] = -1
    p, s = _run_grouped(bsq, "nvfp4", d, 1, ridx=ridx, expert_ids=eid, expect_error=0 if skipped else 4,
                        kernel="token")
    safe = np.where((ridx < 0) | (ridx >= 600), 0, ridx)
    p_ref, pw, s_ref, sw = oracle.grouped_quantize("nvfp4", d["x_bits"], d["row_offsets"], d["scales_offsets"], eid,
                                                   d["sf_tensor"], safe)
    good = pw.copy()
    good[bad] = False
    np.testing.assert_array_equal(p[good], p_ref[good])
    assert np.all(p[bad] == SENTINEL)
    assert np.all(p[~pw] == SENTINEL)
    assert bsq.device_error() == 0


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
def test_token_kernel_full_buckets_many_tokens_per_block(bsq, fmt):
    """More than 16 tokens per block (warps take whole tokens rather than
    shared (token, step) units) with one source row in 40 positions, one in
    exactly 16 and one in 17, and row_indices 4 bytes past a 16-byte
    boundary: the re-scan of the static path, against the oracle."""
    d = wl.config_grouped_prefill(seed=23, tokens=4000, K=32, num_experts=8, top_k=3, fmt=fmt)
    rng = np.random.Generator(np.random.PCG64(24))
    ridx = d["row_indices"].copy()
    ridx[np.isin(ridx, [7, 11, 13])] = 5
    n = ridx.size
    pos = rng.permutation(np.arange(3, n - 3))
    ridx[np.concatenate([[0, 1, 2, n - 3, n - 2, n - 1], pos[:34]])] = 7
    ridx[pos[34:50]] = 11
    ridx[pos[50:67]] = 13
    dev = i32_device(np.concatenate([[0, 0, 0, 0, 7], ridx]))[5:]   # 20 bytes into a 16-byte aligned buffer
    assert dev.data_ptr() % 16 == 4
    total_rows, tsr = d["total_rows"], d["total_scale_rows"]
    ofull, out = guarded(total_rows * oracle.packed_row_bytes(fmt, 32))
    sfull, sc = guarded(oracle.scales5d_bytes(tsr, 32 // oracle.block_size(fmt)))
    bsq.grouped_quantize(to_device_bf16(d["x_bits"]), fmt, u32_device(d["row_offsets"]),
                         u32_device(d["scales_offsets"]), i32_device(d["expert_ids"]),
                         torch.from_numpy(d["sf_tensor"]).cuda() if fmt == "nvfp4" else None, dev,
                         total_rows=total_rows, total_scale_rows=tsr, k_tiles_per_block=1, out=out, scales=sc,
                         kernel="token")
    assert bsq.device_error() == 0
    assert margin_intact(ofull) and margin_intact(sfull)
    _compare(fmt, d, out.cpu().numpy().reshape(total_rows, -1), sc.cpu().numpy(), ridx=ridx)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("kernel", ["stream", "latency", "token", "auto"])
@pytest.mark.parametrize("tokens", [67, 4000])
def test_grouped_workspace_every_kernel(bsq, fmt, kernel, tokens):
    """The scale-staging workspace with every kernel choice (the streaming
    and latency kernels ignore it) on top-3 routing with 67 tokens (the
    token kernel's (token, step) units) and 4000 tokens (whole tokens per
    warp): bytes equal the oracle, padding rows keep their sentinel."""
    d = wl.config_grouped_prefill(seed=31 + tokens, tokens=tokens, K=192, num_experts=12, top_k=3, fmt=fmt)
    p, s = _run_grouped(bsq, fmt, d, 4, kernel=kernel, workspace=True)
    _compare(fmt, d, p, s)


def test_grouped_workspace_bad_source_rows_reported(bsq):
    """With the workspace, a source row outside x in a kept group is still
    reported (BSQ_ERR_VALUE) and its packed row left untouched; every other
    row equals the oracle."""
    d = wl.config_grouped_prefill(seed=8, tokens=40, K=128, num_experts=8, top_k=2)
    ridx = d["row_indices"].copy()
    bad = [3, len(ridx) - 1]
    ridx[bad[0]] = 10_000_000
    ridx[bad[1]] = -5
    p, s = _run_grouped(bsq, "nvfp4", d, 1, ridx=ridx, expect_error=4, kernel="token", workspace=True)
    p_ref, pw, _, _ = oracle.grouped_quantize("nvfp4", d["x_bits"], d["row_offsets"], d["scales_offsets"],
                                              d["expert_ids"], d["sf_tensor"], np.where(ridx < 0, 0, np.minimum(ridx, 39)))
    good = np.ones(d["total_rows"], bool)
    good[bad] = False
    np.testing.assert_array_equal(p[good], p_ref[good])
    assert np.all(p[bad] == SENTINEL)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8", "mxfp4"])
def test_grouped_stream_split_runs_gathered_K7168(bsq, fmt):
    """The streaming kernel on a gathered 8192-row routing (1024 tokens,
    top-8 of 256 experts, K = 7168): few rows, so each block's run of
    columns is split into seven; every written byte against the oracle."""
    d = wl.config_grouped_prefill(seed=11, tokens=1024, K=7168, fmt=fmt)
    p, s = _run_grouped(bsq, fmt, d, 0, kernel="stream")
    _compare(fmt, d, p, s)
