"""The grouped quantize without a gather (row_indices NULL, destination row d
reads source row d): every written byte against the oracle, the rows of
skipped groups, the padding rows of partial 5D bands and the rows past
row_offsets[G] untouched, on the streaming kernel, whose column runs are
split when there are few rows (K = 1120: two runs; the 8192-row case:
seven), and on the library's choice."""
import numpy as np
import pytest

import oracle
import workloads as wl
from bsq_testlib import SENTINEL, guarded, i32_device, margin_intact, to_device_bf16, u32_device
from test_gpu_grouped import _compare, _prefill_reference, _run_grouped

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def bsq():
    import fp8_activation_quantization_bsq_gb300 as m
    from fp8_activation_quantization_bsq_gb300 import _build
    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def _groups(rng, m, K, fmt, n_exp=None, sf=None, trailing=0, in_rows=None):
    """Grouped metadata for group sizes m (no gather): x has a row per
    destination row (or in_rows rows)."""
    G = m.size
    ro = np.concatenate([[0], np.cumsum(m)]).astype(np.uint32)
    so = np.concatenate([[0], np.cumsum(-(-m // 128) * 128)]).astype(np.uint32)
    total_rows = int(ro[-1]) + trailing
    n_exp = G if n_exp is None else n_exp
    eid = np.arange(G, dtype=np.int32) % n_exp
    if sf is None:
        sf = (rng.random(n_exp).astype(np.float32) + np.float32(0.25))
    x = wl.dense_activations(rng, total_rows if in_rows is None else in_rows, K, "blocklognormal")
    return dict(x_bits=x, row_offsets=ro, scales_offsets=so, expert_ids=eid, sf_tensor=sf, row_indices=None,
                total_rows=total_rows, total_scale_rows=int(so[-1]), G=G)


@pytest.mark.parametrize("kernel", ["stream", "auto"])
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("K", [32, 96, 256, 1120])
def test_nogather_group_shapes(bsq, fmt, K, kernel):
    """Empty groups, single rows, a full band, 129 and 300 rows (partial
    last bands), rows past row_offsets[G], K not a multiple of 64."""
    rng = np.random.Generator(np.random.PCG64(K))
    m = np.array([0, 5, 0, 128, 129, 1, 0, 300, 40, 0, 7], np.int64)
    d = _groups(rng, m, K, fmt, trailing=9)
    p, s = _run_grouped(bsq, fmt, d, 0, use_ridx=False, kernel=kernel)
    owned = int(d["row_offsets"][-1])
    _compare(fmt, d, p[:owned], s, use_ridx=False, x_bits=d["x_bits"][:owned])
    assert np.all(p[owned:] == SENTINEL)


@pytest.mark.parametrize("kernel", ["stream", "latency"])
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
def test_nogather_exhaustive_amax_and_extreme_scales(bsq, fmt, kernel):
    """Every BF16 block amax, in groups whose NVFP4 tensor scales span the
    factor table's exact range and beyond (the division path)."""
    from test_gpu_dense import _amax_sweep_matrix
    SF = oracle.block_size(fmt)
    mat = _amax_sweep_matrix(SF, per_row_blocks=16)  # 2040 rows x 16 blocks
    rows = mat.shape[0]
    rng = np.random.Generator(np.random.PCG64(78))
    G = 12
    cuts = np.sort(rng.choice(np.arange(1, rows), G - 1, replace=False))
    m = np.diff(np.concatenate([[0], cuts, [rows]]))
    sf = np.array([1e-37, 2.0 ** -117, 2.0 ** -118, 3e36, 2.0 ** 118, 2.0 ** 119, 6e-36, 1.0, 1e-44, 3.4e38,
                   0.6640316, 2688.0], np.float32)
    d = _groups(rng, m, mat.shape[1], fmt, sf=sf)
    d["x_bits"] = mat
    p, s = _run_grouped(bsq, fmt, d, 0, use_ridx=False, kernel=kernel)
    _compare(fmt, d, p, s, use_ridx=False)


@pytest.mark.parametrize("kernel", ["stream", "latency"])
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8"])
def test_nogather_skipped_groups(bsq, fmt, kernel):
    rng = np.random.Generator(np.random.PCG64(5))
    m = rng.integers(0, 300, size=20)
    d = _groups(rng, m, 256, fmt, n_exp=7)
    eid = d["expert_ids"].copy()
    eid[::3] = -1
    p, s = _run_grouped(bsq, fmt, d, 0, use_ridx=False, expert_ids=eid, kernel=kernel)
    _compare(fmt, d, p, s, use_ridx=False, expert_ids=eid)


@pytest.mark.parametrize("kernel", ["stream", "latency"])
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
def test_nogather_strided_input_and_16_byte_aligned_outputs(bsq, fmt, kernel):
    """Input rows K + 8 elements apart and packed / scale outputs 16 bytes
    past a 32-byte boundary (16-byte stores)."""
    rng = np.random.Generator(np.random.PCG64(6))
    K = 288
    d = _groups(rng, np.array([130, 3, 257, 64], np.int64), K, fmt)
    rows = d["x_bits"].shape[0]
    wide = np.zeros((rows, K + 8), np.uint16)
    wide[:, :K] = d["x_bits"]
    wide[:, K:] = 0x7F00  # huge values outside the view
    x = to_device_bf16(wide)[:, :K]
    total_rows, tsr = d["total_rows"], d["total_scale_rows"]
    ob = total_rows * oracle.packed_row_bytes(fmt, K)
    sb = oracle.scales5d_bytes(tsr, K // oracle.block_size(fmt))
    ofull, _ = guarded(ob + 16)
    sfull, _ = guarded(sb + 16)
    out, sc = ofull[16:16 + ob], sfull[16:16 + sb]
    bsq.grouped_quantize(x, fmt, u32_device(d["row_offsets"]), u32_device(d["scales_offsets"]),
                         i32_device(d["expert_ids"]),
                         torch.from_numpy(d["sf_tensor"]).cuda() if fmt == "nvfp4" else None, None,
                         total_rows=total_rows, total_scale_rows=tsr, out=out, scales=sc, kernel=kernel)
    assert bsq.device_error() == 0
    assert margin_intact(ofull) and margin_intact(sfull)
    assert np.all(ofull[:16].cpu().numpy() == SENTINEL) and np.all(sfull[:16].cpu().numpy() == SENTINEL)
    _compare(fmt, d, out.cpu().numpy().reshape(total_rows, -1), sc.cpu().numpy(), use_ridx=False)


@pytest.mark.parametrize("kernel", ["stream", "latency"])
def test_nogather_source_rows_past_x_are_reported(bsq, kernel):
    """x shorter than the destination rows: the rows past x are reported
    (BSQ_ERR_VALUE) and left unwritten, every other row exact."""
    rng = np.random.Generator(np.random.PCG64(7))
    m = np.array([100, 200, 60], np.int64)
    d = _groups(rng, m, 128, "nvfp4", in_rows=250)
    p, s = _run_grouped(bsq, "nvfp4", d, 0, use_ridx=False, kernel=kernel, expect_error=4)
    x_full = np.zeros((d["total_rows"], 128), np.uint16)
    x_full[:250] = d["x_bits"]
    p_ref, pw, _, _ = oracle.grouped_quantize("nvfp4", x_full, d["row_offsets"], d["scales_offsets"],
                                              d["expert_ids"], d["sf_tensor"], None)
    np.testing.assert_array_equal(p[:250][pw[:250]], p_ref[:250][pw[:250]])
    assert np.all(p[250:] == SENTINEL)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8", "mxfp4"])
@pytest.mark.parametrize("kernel", ["auto"])
def test_nogather_prefill_full_size(bsq, fmt, kernel):
    """The 32768-row prefill groups with their rows already permuted (the
    gathered token rows as x), K = 7168: every packed row and written scale
    byte against the oracle, the padding scale rows untouched."""
    d, (chunks, refs) = _prefill_reference(fmt)
    xg = d["x_bits"][d["row_indices"]]
    dn = dict(d, x_bits=xg, row_indices=None)
    p, s = _run_grouped(bsq, fmt, dn, 0, use_ridx=False, kernel=kernel)
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


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8", "mxfp4"])
def test_nogather_split_runs_K7168(bsq, fmt):
    """8192 rows of 7168 columns (1024 tokens, top-8 of 256 experts, rows
    already permuted): the streaming kernel splits each block's run of
    columns into seven; every written byte against the oracle."""
    d = wl.config_grouped_prefill(seed=11, tokens=1024, K=7168, fmt=fmt)
    d = dict(d, x_bits=d["x_bits"][d["row_indices"]], row_indices=None)
    p, s = _run_grouped(bsq, fmt, d, 0, use_ridx=False, kernel="stream")
    _compare(fmt, d, p, s, use_ridx=False)
