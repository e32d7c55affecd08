"""The per-expert tensor-scale entry point that allocates nothing.

bsq_grouped_tensor_sf_noalloc serves callers that cannot obtain device memory
where they need the scales (a plugin interface that passes only input and
output buffers, a framework that owns all device memory through its own pool,
a loop that cannot take cudaMalloc's synchronization): its scratch is a static
array inside the library, shared by every call on a device.  These tests call
it through the C ABI and compare it with bsq_grouped_tensor_sf, which takes a
caller-allocated workspace, bit for bit (the scales are exact), on calls in a
row whose inputs differ so that anything left over from the previous call
would show.  The file sorts last so that a run stopping at the first failure
has run every other test; it builds and loads the library itself, so it also
passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import workloads as wl
from bsq_testlib import i32_device, to_device_bf16, u32_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

MAX_EXPERTS = 1024   # BSQ_NOALLOC_MAX_EXPERTS in include/bsq.h
SHAPE, VALUE = 2, 4


@pytest.fixture(scope="module")
def lib():
    from fp8_activation_quantization_bsq_gb300 import _build
    import fp8_activation_quantization_bsq_gb300 as bsq
    _build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return bsq.lib()


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _case(seed, tokens, K, E, top_k, scale):
    d = wl.config_grouped_prefill(seed=seed, tokens=tokens, K=K, num_experts=E, top_k=top_k)
    x = wl.f32_to_bf16_bits(wl.bf16_bits_to_f32(d["x_bits"]) * np.float32(scale))
    return dict(x=to_device_bf16(x), ro=u32_device(d["row_offsets"]), eid=i32_device(d["expert_ids"]),
                ridx=i32_device(d["row_indices"]), G=int(d["G"]), total_rows=int(d["total_rows"]), E=E)


def _noalloc(lib, c, num_experts=None):
    E = c["E"] if num_experts is None else num_experts
    sf = torch.full((E,), -1.0, dtype=torch.float32, device="cuda")
    x = c["x"]
    rc = lib.bsq_grouped_tensor_sf_noalloc(_p(x), x.shape[0], x.shape[1], x.stride(0), _p(c["ro"]),
                                           _p(c["eid"]), _p(c["ridx"]), c["G"], c["total_rows"],
                                           _p(sf), E, _stream())
    return rc, sf


def _with_workspace(lib, c):
    E = c["E"]
    sf = torch.full((E,), -1.0, dtype=torch.float32, device="cuda")
    ws = torch.zeros(lib.bsq_grouped_tensor_sf_workspace_bytes(E), dtype=torch.uint8, device="cuda")
    x = c["x"]
    rc = lib.bsq_grouped_tensor_sf(_p(x), x.shape[0], x.shape[1], x.stride(0), _p(c["ro"]), _p(c["eid"]),
                                   _p(c["ridx"]), c["G"], c["total_rows"], _p(sf), E, _p(ws), ws.numel(),
                                   _stream())
    assert rc == 0
    return sf


def _device_error(lib):
    code = ctypes.c_int32(0)
    assert lib.bsq_device_error(_stream(), ctypes.byref(code)) == 0
    return code.value


def test_noalloc_matches_workspace_entry_point_on_calls_in_a_row(lib):
    # large values first, then the same routing at 1/1000 the magnitude, then
    # more experts than before: stale maxima or a stale counter would show
    cases = [_case(11, 300, 512, 64, 6, 1.0), _case(11, 300, 512, 64, 6, 1e-3),
             _case(12, 96, 2048, 256, 8, 3.0)]
    for c in cases:
        rc, got = _noalloc(lib, c)
        assert rc == 0
        want = _with_workspace(lib, c)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got.cpu().numpy(), want.cpu().numpy())
        assert _device_error(lib) == 0
    # the same input twice: identical results
    rc1, a = _noalloc(lib, cases[0])
    rc2, b = _noalloc(lib, cases[0])
    assert rc1 == rc2 == 0
    np.testing.assert_array_equal(a.cpu().numpy(), b.cpu().numpy())


def test_noalloc_at_the_expert_limit(lib):
    c = _case(13, 256, 256, MAX_EXPERTS, 8, 1.0)
    rc, got = _noalloc(lib, c)
    assert rc == 0
    np.testing.assert_array_equal(got.cpu().numpy(), _with_workspace(lib, c).cpu().numpy())
    assert _device_error(lib) == 0


def test_noalloc_rejects_sizes_beyond_the_limit(lib):
    c = _case(14, 16, 256, 8, 2, 1.0)
    rc, sf = _noalloc(lib, c, num_experts=MAX_EXPERTS + 1)
    assert rc == SHAPE
    assert np.all(sf.cpu().numpy() == -1.0)          # nothing was enqueued
    rc, _ = _noalloc(lib, c, num_experts=0)
    assert rc == VALUE
