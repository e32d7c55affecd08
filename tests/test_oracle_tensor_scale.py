"""Pins of the oracle's tensor scales (CPU only): closed forms on hand-picked
tensors, the link to the block scale (the global-amax block lands on the
E4M3 maximum), and the per-expert reduction against per-expert dense calls."""
import numpy as np

import oracle
import workloads as wl


def _bits(vals):
    return wl.f32_to_bf16_bits(np.array(vals, dtype=np.float32))


def test_tensor_sf_closed_forms():
    a, s = oracle.tensor_sf(_bits([[0.0, -2688.0], [1.0, 3.0]]))
    assert a == 2688.0 and s == 1.0
    a, s = oracle.tensor_sf(_bits([[0.5, -2.0]]))
    assert a == 2.0 and s == 1344.0
    a, s = oracle.tensor_sf(_bits([[0.0, -0.0]]))
    assert a == 0.0 and s == 1.0
    a, s = oracle.tensor_sf(np.zeros((0, 32), np.uint16))
    assert a == 0.0 and s == 1.0
    a, s = oracle.tensor_sf(_bits([[3.0]]))
    assert s == np.float32(896.0)
    # inexact quotient: one FP32 rounding of 2688 / 7
    a, s = oracle.tensor_sf(_bits([[7.0]]))
    assert s == np.float32(np.float32(2688) / np.float32(7))
    # magnitude ignores the sign, including the sign of the largest value
    assert oracle.tensor_sf(_bits([[-5.0, 4.0]]))[0] == 5.0


def test_tensor_sf_puts_the_largest_block_on_448():
    for seed in range(3):
        c = wl.config_dense_nvfp4_large(seed=seed, M=32, K=512)
        amax, tsf = oracle.tensor_sf(c["x_bits"])
        xf = np.abs(wl.bf16_bits_to_f32(c["x_bits"]))
        assert amax == xf.max()
        _, sc = oracle.quantize_rank2("nvfp4", c["x_bits"], tsf)
        blk = np.unravel_index(np.argmax(xf.reshape(32, -1, 16).max(-1)), sc.shape)
        assert sc[blk] == 0x7E


def test_expert_tensor_sf_matches_per_expert_tensor_sf():
    d = wl.config_grouped_prefill(seed=2, tokens=48, K=128, num_experts=12, top_k=3)
    amax, sf = oracle.expert_tensor_sf(d["x_bits"], d["row_offsets"], d["expert_ids"], 12,
                                       d["row_indices"])
    ro = d["row_offsets"].astype(int)
    seen = set()
    for g, e in enumerate(d["expert_ids"]):
        rows = d["row_indices"][ro[g]:ro[g + 1]]
        a, s = oracle.tensor_sf(d["x_bits"][rows])
        assert amax[e] == a and sf[e] == s
        seen.add(int(e))
    for e in set(range(12)) - seen:
        assert amax[e] == 0 and sf[e] == 1.0
    # the workloads' per-expert sf (computed independently) agrees
    np.testing.assert_array_equal(sf, d["sf_tensor"])


def test_expert_tensor_sf_skips_negative_ids_and_merges_repeated_experts():
    x = _bits([[1.0, 0.0], [-8.0, 2.0], [0.5, 0.25], [3.0, -1.0]])
    amax, sf = oracle.expert_tensor_sf(x, [0, 1, 2, 4], [1, -1, 1], 3)
    assert amax[1] == 3.0 and amax[0] == 0 and amax[2] == 0
    assert sf[1] == np.float32(896.0) and sf[0] == 1.0
