"""Pins of the oracle's block quantizers, 5D layout, grouped driver and
consumer check (CPU only).

Hand-worked blocks come from ``tests/golden/hand_worked_blocks.json`` (derived
by hand from the format definitions and the block-scale readings of the
quantize_dynamic_scaled_async_fp4_kernel page).  The rest are closed forms,
invariants that any correct implementation satisfies, and reductions of the
grouped kernel (grouped_quantize_dynamic_scaled_fp4_async_kernel page) and
the reinterleave (block_scales_interleave, module index) to the dense case.
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_blocks.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)["blocks"]


@pytest.mark.parametrize("blk", _golden(), ids=lambda b: b["name"])
def test_hand_worked_block(blk):
    fmt = blk["fmt"]
    SF = oracle.block_size(fmt)
    x = np.zeros((1, SF), dtype=np.uint16)
    for i, h in enumerate(blk["x_bf16"]):
        x[0, i] = int(h, 16)
    packed, scales = oracle.quantize_rank2(fmt, x, np.float32(blk["tensor_sf"]))
    assert scales.shape == (1, 1)
    assert scales[0, 0] == int(blk["scale_byte"], 16)
    want = bytes.fromhex(blk["packed_hex"])
    row = packed[0].tobytes()
    assert row[: len(want)] == want
    assert row[len(want):] == bytes(len(row) - len(want))


# ---- 5D layout ----------------------------------------------------------

def test_offset_5d_hand_checked_entries():
    Kt = 3
    cases = {(0, 0): 0, (1, 0): 16, (31, 0): 496, (32, 0): 4, (64, 0): 8, (96, 0): 12,
             (33, 2): 16 + 4 + 2, (127, 3): 511, (0, 1): 1, (0, 4): 512, (0, 11): 2 * 512 + 3,
             (128, 0): Kt * 512, (129, 5): Kt * 512 + 512 + 16 + 1}
    for (m, s), off in cases.items():
        assert oracle.offset_5d(m, s, Kt) == off, (m, s)


@pytest.mark.parametrize("Mt,Kt", [(1, 1), (2, 3), (3, 2)])
def test_offset_5d_is_a_bijection(Mt, Kt):
    m, s = np.meshgrid(np.arange(Mt * 128), np.arange(Kt * 4), indexing="ij")
    off = oracle.offset_5d(m, s, Kt).ravel()
    np.testing.assert_array_equal(np.sort(off), np.arange(Mt * Kt * 512))


@pytest.mark.parametrize("M,S", [(1, 1), (127, 5), (128, 4), (129, 9), (300, 14)])
def test_5d_scatter_matches_reshape_view(M, S):
    rng = np.random.Generator(np.random.PCG64(M * 100 + S))
    sc = rng.integers(1, 256, size=(M, S), dtype=np.uint8)
    buf = oracle.scales_to_5d(sc)
    assert buf.size == oracle.scales5d_bytes(M, S)
    view = oracle.scales_from_5d_view(buf, M, S)
    np.testing.assert_array_equal(view[:M, :S], sc)
    assert not view[M:, :].any() and not view[:, S:].any()


def test_interleave_is_a_permutation_with_zero_padding():
    rng = np.random.Generator(np.random.PCG64(3))
    M, S, ld = 200, 10, 16
    raw = rng.integers(1, 256, size=(M, ld), dtype=np.uint8)
    out = oracle.scales_interleave(raw, M, S, ld)
    want = np.concatenate([raw[:, :S].ravel(), np.zeros(out.size - M * S, np.uint8)])
    np.testing.assert_array_equal(np.sort(out), np.sort(want))
    np.testing.assert_array_equal(oracle.scales_from_5d_view(out, M, S)[:M, :S], raw[:, :S])


def test_interleave_equals_quantize_scales():
    c = wl.config_dense_nvfp4_small()
    _, s2 = oracle.quantize_rank2("nvfp4", c["x_bits"], c["tensor_sf"])
    _, s5 = oracle.quantize("nvfp4", c["x_bits"], c["tensor_sf"])
    np.testing.assert_array_equal(oracle.scales_interleave(s2, *s2.shape, s2.shape[1]), s5)


# ---- invariants of the block scales -------------------------------------

def _rand_bf16(seed, M, K, kind="blocklognormal"):
    return wl.dense_activations(np.random.Generator(np.random.PCG64(seed)), M, K, kind)


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp8"])
def test_mx_scale_power_of_two_and_no_headroom_waste(fmt):
    x = _rand_bf16(21, 64, 1024)
    packed, sc = oracle.quantize_rank2(fmt, x)
    xf = wl.bf16_bits_to_f32(x).astype(np.float64).reshape(64, -1, 32)
    amax = np.abs(xf).max(-1)
    e = sc.astype(np.int64) - 127
    qmax = 6.0 if fmt == "mxfp4" else 448.0
    r = amax * np.ldexp(1.0, -e)
    nz = amax > 0
    eps = 2.0 ** -23
    assert np.all(r[nz] > qmax / 2 * (1 - eps)) and np.all(r[nz] <= qmax * (1 + eps))
    assert np.all(sc[~nz] == 0)


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp8"])
def test_mx_dequant_error_bound(fmt):
    x = _rand_bf16(22, 64, 1024)
    packed, sc = oracle.quantize_rank2(fmt, x)
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    deq = oracle.dequantize(fmt, packed, sc)
    scale = np.repeat(oracle.e8m0_decode(sc), 32, axis=1)
    y = np.abs(xf) / scale                          # |x| in element units
    mags = oracle.E2M1_MAGNITUDES if fmt == "mxfp4" else oracle.E4M3_MAGNITUDES
    idx = np.clip(np.searchsorted(mags, y), 1, len(mags) - 1)
    half_gap = (mags[idx] - mags[idx - 1]) / 2
    sat = np.maximum(y - mags[-1], 0)              # only the FP32 rounding sliver
    assert np.all(sat <= mags[-1] * 2.0 ** -22)
    assert np.all(np.abs(xf - deq) <= (half_gap + sat) * scale * (1 + 2.0 ** -20))


def test_nvfp4_global_amax_block_gets_max_scale():
    for seed in range(5):
        c = wl.config_dense_nvfp4_small(seed=seed)
        xf = np.abs(wl.bf16_bits_to_f32(c["x_bits"])).reshape(c["M"], -1, 16)
        _, sc = oracle.quantize_rank2("nvfp4", c["x_bits"], c["tensor_sf"])
        blk = np.unravel_index(np.argmax(xf.max(-1)), sc.shape)
        assert sc[blk] == 0x7E


def test_nvfp4_dequant_error_bound():
    c = wl.config_dense_nvfp4_large(M=64, K=1024)
    packed, sc = oracle.quantize_rank2("nvfp4", c["x_bits"], c["tensor_sf"])
    xf = wl.bf16_bits_to_f32(c["x_bits"]).astype(np.float64)
    deq = oracle.dequantize("nvfp4", packed, sc, c["tensor_sf"])
    ds = oracle.e4m3_decode(sc)
    unit = np.repeat(ds / np.float64(c["tensor_sf"]), 16, axis=1)
    normal = np.repeat(ds >= 2.0 ** -6, 16, axis=1)
    err = np.abs(xf - deq)
    assert np.all(err[normal] <= unit[normal] * (1 + 2.0 ** -20))
    zero = np.repeat(ds == 0, 16, axis=1)
    assert np.all(deq[zero] == 0)


def test_nvfp4_power_of_two_rescaling_invariance():
    # scaling x by 2^k and tensor_sf by 2^-k leaves every byte unchanged
    c = wl.config_dense_nvfp4_large(M=32, K=512)
    xf = wl.bf16_bits_to_f32(c["x_bits"])
    p0, s0 = oracle.quantize_rank2("nvfp4", c["x_bits"], c["tensor_sf"])
    for k in (-3, 5):
        xk = wl.f32_to_bf16_bits(xf * np.float32(2.0 ** k))
        pk, sk = oracle.quantize_rank2("nvfp4", xk, np.float32(c["tensor_sf"] * np.float32(2.0 ** -k)))
        np.testing.assert_array_equal(pk, p0)
        np.testing.assert_array_equal(sk, s0)


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp8"])
def test_mx_power_of_two_rescaling_shifts_scale_only(fmt):
    x = _rand_bf16(23, 16, 256, "normal")
    xf = wl.bf16_bits_to_f32(x)
    p0, s0 = oracle.quantize_rank2(fmt, x)
    for k in (-7, 9):
        pk, sk = oracle.quantize_rank2(fmt, wl.f32_to_bf16_bits(xf * np.float32(2.0 ** k)))
        np.testing.assert_array_equal(pk, p0)
        np.testing.assert_array_equal(sk.astype(int), s0.astype(int) + k)


# ---- consumer check: dequantise-then-dot through the 5D layout -----------

@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
def test_naive_matmul_through_5d_matches_rank2(fmt):
    rng = np.random.Generator(np.random.PCG64(31))
    M, N, K = 130, 40, 256
    a = wl.dense_activations(rng, M, K, "blocklognormal")
    b = wl.dense_activations(rng, N, K, "blocklognormal")
    ta = wl.tensor_sf_from_amax(np.abs(wl.bf16_bits_to_f32(a)).max()) if fmt == "nvfp4" else 1.0
    tb = wl.tensor_sf_from_amax(np.abs(wl.bf16_bits_to_f32(b)).max()) if fmt == "nvfp4" else 1.0
    pa, sa = oracle.quantize_rank2(fmt, a, ta)
    pb, sb = oracle.quantize_rank2(fmt, b, tb)
    c5 = oracle.naive_block_scaled_matmul(fmt, pa, oracle.scales_to_5d(sa), ta,
                                          pb, oracle.scales_to_5d(sb), tb, K)
    c2 = oracle.dequantize(fmt, pa, sa, ta) @ oracle.dequantize(fmt, pb, sb, tb).T
    np.testing.assert_array_equal(c5, c2)
    # the product approximates the BF16 product
    ref = wl.bf16_bits_to_f32(a).astype(np.float64) @ wl.bf16_bits_to_f32(b).astype(np.float64).T
    rel = np.linalg.norm(c5 - ref) / np.linalg.norm(ref)
    assert rel < (0.5 if fmt != "mxfp8" else 0.15)
    # swapping two blocks' scale bytes in the 5D buffer changes the product
    s5 = oracle.scales_to_5d(sa)
    i, j = oracle.offset_5d(1, 0, -(-sa.shape[1] // 4)), oracle.offset_5d(40, 1, -(-sa.shape[1] // 4))
    assert s5[i] != s5[j]
    s5[i], s5[j] = s5[j], s5[i]
    c_sw = oracle.naive_block_scaled_matmul(fmt, pa, s5, ta, pb, oracle.scales_to_5d(sb), tb, K)
    assert not np.array_equal(c_sw, c5)


# ---- grouped reduces to dense ---------------------------------------------

@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
def test_grouped_single_group_identity_equals_dense(fmt):
    c = wl.config_dense_nvfp4_small()
    M = c["M"]
    sf = np.array([c["tensor_sf"]], dtype=np.float32)
    p, pw, s5, sw = oracle.grouped_quantize(fmt, c["x_bits"], [0, M], [0, 128], [0], sf)
    pd, s5d = oracle.quantize(fmt, c["x_bits"], c["tensor_sf"])
    assert pw.all() and sw.all()
    np.testing.assert_array_equal(p, pd)
    np.testing.assert_array_equal(s5, s5d)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8"])
def test_grouped_equals_per_expert_dense(fmt):
    d = wl.config_grouped_prefill(seed=7, tokens=64, K=256, num_experts=16, top_k=4, fmt=fmt)
    p, pw, s5, sw = oracle.grouped_quantize(fmt, d["x_bits"], d["row_offsets"], d["scales_offsets"],
                                            d["expert_ids"], d["sf_tensor"], d["row_indices"])
    assert pw.all()
    S = 256 // oracle.block_size(fmt)
    view = oracle.scales_from_5d_view(s5, d["total_scale_rows"], S)
    written = oracle.scales_from_5d_view(sw.astype(np.uint8), d["total_scale_rows"], S).astype(bool)
    ro, so = d["row_offsets"].astype(int), d["scales_offsets"].astype(int)
    for g, e in enumerate(d["expert_ids"]):
        rows = d["row_indices"][ro[g]:ro[g + 1]]
        pd, sd = oracle.quantize_rank2(fmt, d["x_bits"][rows], d["sf_tensor"][e])
        np.testing.assert_array_equal(p[ro[g]:ro[g + 1]], pd)
        np.testing.assert_array_equal(view[so[g]:so[g] + len(rows), :S], sd)
        assert written[so[g]:so[g] + len(rows)].all()
        assert not written[so[g] + len(rows):so[g + 1]].any()      # padding rows untouched


def test_grouped_skips_negative_expert_and_honours_row_indices():
    rng = np.random.Generator(np.random.PCG64(8))
    x = wl.dense_activations(rng, 10, 64, "normal")
    ro, so = [0, 3, 5, 9], [0, 128, 256, 384]
    eid = [2, -1, 0]
    sf = np.array([1.5, 7.0, 3.0], dtype=np.float32)
    ridx = np.array([9, 0, 4, 1, 1, 8, 7, 6, 5], dtype=np.int32)
    p, pw, s5, sw = oracle.grouped_quantize("nvfp4", x, ro, so, eid, sf, ridx)
    np.testing.assert_array_equal(pw, [1, 1, 1, 0, 0, 1, 1, 1, 1])
    pd, _ = oracle.quantize_rank2("nvfp4", x[[9, 0, 4]], sf[2])
    np.testing.assert_array_equal(p[:3], pd)
    pd, _ = oracle.quantize_rank2("nvfp4", x[[8, 7, 6, 5]], sf[0])
    np.testing.assert_array_equal(p[5:], pd)
    assert not p[3:5].any()
    view_w = oracle.scales_from_5d_view(sw.astype(np.uint8), 384, 4).astype(bool)
    assert view_w[0:3].all() and not view_w[3:128].any() and not view_w[128:256].any()
    assert view_w[256:260].all() and not view_w[260:].any()
