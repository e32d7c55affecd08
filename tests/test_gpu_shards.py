"""The path partitions with no exchange: quantizing shards one after the
other (as separate ranks would) reproduces the unsharded outputs byte for
byte.  Dense tensors split on 128-row boundaries (each shard's 5D scales
are a contiguous slice of the whole buffer); grouped work splits by groups
(expert-parallel), each shard with its own rebased metadata writing into its
slice of the outputs.  The one exchange a sharded tensor needs -- a global
NVFP4 tensor_sf -- reduces to the maximum of the shards' amax."""
import numpy as np
import pytest

import oracle
import workloads as wl
from bsq_testlib import i32_device, to_device_bf16, u32_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def bsq():
    import fp8_activation_quantization_bsq_gb300 as m
    from fp8_activation_quantization_bsq_gb300 import _build
    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("shards", [2, 3])
def test_dense_row_shards_equal_the_whole(bsq, fmt, shards):
    rng = np.random.Generator(np.random.PCG64(41))
    M, K = 128 * 5 + 40, 1056
    bits = wl.dense_activations(rng, M, K, "rowlognormal")
    x = to_device_bf16(bits)
    amax, tsf = oracle.tensor_sf(bits)
    tsf = float(tsf) if fmt == "nvfp4" else 1.0
    whole_p, whole_s = bsq.quantize(x, fmt, tsf)
    # shard on 128-row boundaries
    tiles = -(-M // 128)
    cuts = [min(M, 128 * (tiles * i // shards)) for i in range(shards + 1)]
    out = torch.empty_like(whole_p)
    sc = torch.empty_like(whole_s)
    S = K // oracle.block_size(fmt)
    band = -(-S // 4) * 512                          # 5D bytes per 128-row band
    for r0, r1 in zip(cuts[:-1], cuts[1:]):
        bsq.quantize(x[r0:r1], fmt, tsf, out=out[r0:r1],
                     scales=sc[(r0 // 128) * band:(-(-r1 // 128)) * band])
    assert torch.equal(out, whole_p) and torch.equal(sc, whole_s)
    # global tensor scale = f(max of the shards' amax)
    shard_amax = [float(bsq.tensor_sf(x[r0:r1])[0]) for r0, r1 in zip(cuts[:-1], cuts[1:])]
    assert max(shard_amax) == float(amax)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8"])
def test_grouped_expert_shards_equal_the_whole(bsq, fmt):
    d = wl.config_grouped_prefill(seed=12, tokens=300, K=512, num_experts=16, top_k=4)
    ro, so = d["row_offsets"].astype(np.int64), d["scales_offsets"].astype(np.int64)
    eid, ridx, G = d["expert_ids"], d["row_indices"], d["G"]
    x = to_device_bf16(d["x_bits"])
    sf = torch.from_numpy(d["sf_tensor"]).cuda() if fmt == "nvfp4" else None
    whole_p, whole_s = bsq.grouped_quantize(x, fmt, u32_device(ro), u32_device(so), i32_device(eid), sf,
                                            i32_device(ridx), total_rows=d["total_rows"],
                                            total_scale_rows=d["total_scale_rows"], k_tiles_per_block=2)
    K = d["K"]
    rb = oracle.packed_row_bytes(fmt, K)
    band = -(-(K // oracle.block_size(fmt)) // 4) * 512
    out = torch.zeros_like(whole_p)
    sc = torch.zeros_like(whole_s)
    for g0, g1 in ((0, G // 3), (G // 3, G - 2), (G - 2, G)):
        r0, r1, s0, s1 = int(ro[g0]), int(ro[g1]), int(so[g0]), int(so[g1])
        bsq.grouped_quantize(x, fmt, u32_device(ro[g0:g1 + 1] - r0), u32_device(so[g0:g1 + 1] - s0),
                             i32_device(eid[g0:g1]), sf, i32_device(ridx[r0:r1]),
                             total_rows=r1 - r0, total_scale_rows=s1 - s0, k_tiles_per_block=2,
                             out=out.view(-1)[r0 * rb:r1 * rb].view(r1 - r0, rb),
                             scales=sc[(s0 // 128) * band:(s1 // 128) * band])
    assert bsq.device_error() == 0
    p_ref, pw, s_ref, sw = oracle.grouped_quantize(fmt, d["x_bits"], ro, so, eid, d["sf_tensor"], ridx)
    np.testing.assert_array_equal(out.cpu().numpy()[pw], whole_p.cpu().numpy()[pw])
    np.testing.assert_array_equal(sc.cpu().numpy()[sw], whole_s.cpu().numpy()[sw])
    np.testing.assert_array_equal(out.cpu().numpy()[pw], p_ref[pw])
