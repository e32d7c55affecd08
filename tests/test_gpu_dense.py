"""GPU parity of dense quantize and the rank-2 -> 5D reinterleave against the
CPU oracle, through the C ABI (Python binding).  Bit-exact: the outputs are
integer codes and bytes.

Operations: quantize_dynamic_scaled_fp4fp8 / quantize_dynamic_scaled_async_fp4_kernel
and block_scales_interleave (Modular block_scaled_quantization pages).
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from bsq_testlib import guarded, margin_intact, to_device_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
FMTS = ["nvfp4", "mxfp4", "mxfp8"]


@pytest.fixture(scope="module")
def bsq():
    import fp8_activation_quantization_bsq_gb300 as m
    from fp8_activation_quantization_bsq_gb300 import _build
    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def _tsf(fmt, bits):
    if fmt != "nvfp4":
        return np.float32(1.0)
    return wl.tensor_sf_from_amax(np.abs(wl.bf16_bits_to_f32(bits)).max() if bits.size else 0)


def _run_dense(bsq, fmt, bits, tsf, ld=None):
    M, K = bits.shape
    if ld is None:
        x = to_device_bf16(bits)
    else:
        wide = np.zeros((M, ld), dtype=np.uint16)
        wide[:, :K] = bits
        wide[:, K:] = 0x4780  # large values outside the view must not leak in
        x = to_device_bf16(wide)[:, :K]
    ob = M * oracle.packed_row_bytes(fmt, K)
    sb = oracle.scales5d_bytes(M, K // oracle.block_size(fmt))
    ofull, out = guarded(ob)
    sfull, sc = guarded(sb)
    bsq.quantize(x, fmt, float(tsf), out=out, scales=sc)
    assert bsq.device_error() == 0
    assert margin_intact(ofull) and margin_intact(sfull)
    return out.cpu().numpy().reshape(M, -1), sc.cpu().numpy()


SHAPES = [(1, 32), (127, 96), (128, 128), (129, 160), (257, 64), (300, 1056), (64, 7168), (200, 352)]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,K", SHAPES)
def test_dense_ragged_shapes(bsq, fmt, M, K):
    rng = np.random.Generator(np.random.PCG64(M * 7919 + K))
    bits = wl.dense_activations(rng, M, K, "blocklognormal")
    tsf = _tsf(fmt, bits)
    p, s = _run_dense(bsq, fmt, bits, tsf)
    p_ref, s_ref = oracle.quantize(fmt, bits, tsf)
    np.testing.assert_array_equal(p, p_ref)
    np.testing.assert_array_equal(s, s_ref)


@pytest.mark.parametrize("fmt", FMTS)
def test_dense_small_config_exact(bsq, fmt):
    c = wl.config_dense_nvfp4_small()
    tsf = c["tensor_sf"] if fmt == "nvfp4" else 1.0
    p, s = _run_dense(bsq, fmt, c["x_bits"], tsf)
    p_ref, s_ref = oracle.quantize(fmt, c["x_bits"], tsf)
    np.testing.assert_array_equal(p, p_ref)
    np.testing.assert_array_equal(s, s_ref)


@pytest.mark.parametrize("fmt", FMTS)
def test_dense_strided_input(bsq, fmt):
    rng = np.random.Generator(np.random.PCG64(99))
    bits = wl.dense_activations(rng, 150, 192, "rowlognormal")
    tsf = _tsf(fmt, bits)
    p, s = _run_dense(bsq, fmt, bits, tsf, ld=264)
    p_ref, s_ref = oracle.quantize(fmt, bits, tsf)
    np.testing.assert_array_equal(p, p_ref)
    np.testing.assert_array_equal(s, s_ref)


def _edge_matrix():
    """Signed zeros, BF16 extremes (max, min normal, subnormals), element
    midpoints and an all-zero row, 32 x 256."""
    rng = np.random.Generator(np.random.PCG64(4242))
    m = wl.dense_activations(rng, 32, 256, "normal")
    m[0, :] = 0x0000
    m[1, :] = 0x8000
    m[2, ::2] = 0x8000
    m[3, :] = 0x7F7F          # BF16 max
    m[3, 1::3] = 0xFF7F
    m[4, :] = 0x0001          # smallest subnormal
    m[4, 5::7] = 0x8001
    m[5, :] = 0x0080          # smallest normal
    m[6, :16] = 0x7F7F        # huge block next to tiny ones
    m[6, 16:32] = 0x0003
    m[7, :] = np.array([0x3E80, 0x3F40, 0x3FA0, 0x3FE0, 0x4020, 0x4060, 0x40A0, 0x40C0] * 32, np.uint16)
    m[8, :] = 0x40E0          # 7.0 everywhere
    m[9, 0:32] = 0x0000
    m[9, 31] = 0x0001         # a block whose amax is subnormal
    return m


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("tsf", [None, 1.0, 1e-30, 1e30, 1.4e-45])
def test_dense_edge_values(bsq, fmt, tsf):
    bits = _edge_matrix()
    if tsf is None:
        tsf = _tsf("nvfp4", bits)
    if fmt != "nvfp4" and tsf not in (1.0,):
        pytest.skip("tensor_sf only matters for NVFP4")
    p, s = _run_dense(bsq, fmt, bits, tsf)
    p_ref, s_ref = oracle.quantize(fmt, bits, tsf)
    np.testing.assert_array_equal(s, s_ref)
    np.testing.assert_array_equal(p, p_ref)


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp8"])
def test_element_cast_exhaustive_bf16(bsq, fmt):
    """Every BF16 value within the element range, cast with a unit scale:
    each 32-block carries one element equal to Qmax, so e = 0 and x*2^-e = x."""
    qmax = 6.0 if fmt == "mxfp4" else 448.0
    vals = wl.bf16_bits_to_f32(np.arange(1 << 16, dtype=np.uint32).astype(np.uint16))
    keep = np.isfinite(vals) & (np.abs(vals) <= qmax)
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)[keep]
    pad = (-len(bits)) % 31
    bits = np.concatenate([bits, np.zeros(pad, np.uint16)]).reshape(-1, 31)
    top = wl.f32_to_bf16_bits(np.full((bits.shape[0], 1), qmax, np.float32))
    blocks = np.concatenate([top, bits], axis=1)                   # (n, 32)
    n = blocks.shape[0]
    rows = -(-n // 32)
    mat = np.zeros((rows * 32, 32), np.uint16)
    mat[:n] = blocks
    mat = mat.reshape(rows, 32 * 32)
    p, s = _run_dense(bsq, fmt, mat, 1.0)
    p_ref, s_ref = oracle.quantize(fmt, mat, 1.0)
    assert np.all(oracle.scales_from_5d_view(s_ref, rows, 32)[:rows, :32][mat.reshape(rows, 32, 32)[:, :, 0] != 0] == 127)
    np.testing.assert_array_equal(p, p_ref)
    np.testing.assert_array_equal(s, s_ref)


FULL = {
    "nvfp4": lambda: wl.config_dense_nvfp4_large(),
    "mxfp8": lambda: wl.config_dense_mx_wide(fmt="mxfp8"),
    "mxfp4": lambda: wl.config_dense_mx_wide(fmt="mxfp4"),
}


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8", "mxfp4"])
def test_dense_full_size_all_rows(bsq, fmt):
    """The full workloads (NVFP4 8192 x 7168; MXFP8 / MXFP4 16384 x 4096) in
    the benchmark's launch configuration: every packed row and every scale
    byte against the oracle (computed in 512-row chunks over a spawned
    process pool)."""
    from bsq_testlib import oracle_rank2_chunks
    c = FULL[fmt]()
    bits, M, K = c["x_bits"], c["M"], c["K"]
    tsf = c["tensor_sf"]
    p, s = _run_dense(bsq, fmt, bits, tsf)
    refs = oracle_rank2_chunks(fmt, [(bits[r0:r0 + 512], np.float32(tsf)) for r0 in range(0, M, 512)])
    p_ref = np.concatenate([r[0] for r in refs])
    s2 = np.concatenate([r[1] for r in refs])
    np.testing.assert_array_equal(p, p_ref)
    np.testing.assert_array_equal(s, oracle.scales_to_5d(s2))


# ---------------------------------------------------------------- interleave --

@pytest.mark.parametrize("M,S,ld", [(1, 1, 1), (100, 20, 20), (128, 4, 4), (129, 7, 9), (300, 64, 64),
                                    (513, 130, 136), (8192, 448, 448), (77, 200, 203)])
def test_interleave_shapes(bsq, M, S, ld):
    rng = np.random.Generator(np.random.PCG64(M + 31 * S))
    raw = rng.integers(0, 256, size=(M, ld), dtype=np.uint8)
    src = torch.from_numpy(raw).cuda()[:, :S]
    nbytes = oracle.scales5d_bytes(M, S)
    full, out = guarded(nbytes)
    bsq.scales_interleave(src, out=out)
    assert margin_intact(full)
    np.testing.assert_array_equal(out.cpu().numpy(), oracle.scales_interleave(raw, M, S, ld))


def test_interleave_of_quantize_scales(bsq):
    c = wl.config_dense_nvfp4_large(M=1024, K=7168)
    _, s2 = oracle.quantize_rank2("nvfp4", c["x_bits"], c["tensor_sf"])
    _, s5_gpu = _run_dense(bsq, "nvfp4", c["x_bits"], c["tensor_sf"])
    out = bsq.scales_interleave(torch.from_numpy(s2).cuda())
    np.testing.assert_array_equal(out.cpu().numpy(), s5_gpu)


def _amax_sweep_matrix(SF: int, per_row_blocks: int = 64):
    """One block per positive finite BF16 value v (and one zero block):
    elements v, -v, v/3, -v/7 (rounded to BF16) and zeros, so the block amax
    runs over every BF16 magnitude."""
    v = np.arange(0, 0x7F80, dtype=np.uint32).astype(np.uint16)          # +0 .. largest finite
    vf = wl.bf16_bits_to_f32(v)
    n = v.size
    rows = -(-n // per_row_blocks)
    blocks = np.zeros((rows * per_row_blocks, SF), np.uint16)
    blocks[:n, 0] = v
    blocks[:n, 1] = v | 0x8000
    blocks[:n, 2] = wl.f32_to_bf16_bits(vf / np.float32(3.0))
    blocks[:n, 3] = wl.f32_to_bf16_bits(vf / np.float32(-7.0))
    return blocks.reshape(rows, per_row_blocks * SF)


@pytest.mark.parametrize("fmt,tsf", [("mxfp4", 1.0), ("mxfp8", 1.0), ("nvfp4", 1.0),
                                     ("nvfp4", 0.6640316), ("nvfp4", 1e-20), ("nvfp4", 1e20),
                                     ("nvfp4", 2688.0)])
def test_block_scale_exhaustive_amax(bsq, fmt, tsf):
    """Every BF16 block amax -> scale byte and element codes, bit-exact."""
    mat = _amax_sweep_matrix(oracle.block_size(fmt))
    p, s = _run_dense(bsq, fmt, mat, np.float32(tsf))
    p_ref, s_ref = oracle.quantize(fmt, mat, np.float32(tsf))
    np.testing.assert_array_equal(s, s_ref)
    np.testing.assert_array_equal(p, p_ref)
