"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins
catch each of them: the hand-worked blocks and the layout entries must fail
for every mutant, otherwise the pins would not be pinning anything."""
import json
import os

import numpy as np
import pytest

import oracle
import oracle.formats as F
import oracle.layout as L
import oracle.blockquant as Q

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_blocks.json")


def _golden_failures():
    with open(GOLDEN) as f:
        blocks = json.load(f)["blocks"]
    bad = 0
    for blk in blocks:
        SF = Q.block_size(blk["fmt"])
        x = np.zeros((1, SF), dtype=np.uint16)
        for i, h in enumerate(blk["x_bf16"]):
            x[0, i] = int(h, 16)
        p, s = Q.quantize_rank2(blk["fmt"], x, np.float32(blk["tensor_sf"]))
        want = bytes.fromhex(blk["packed_hex"])
        if s[0, 0] != int(blk["scale_byte"], 16) or p[0].tobytes()[: len(want)] != want:
            bad += 1
    return bad


def _ties_away(v, mags, sign_bit):
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v.astype(np.float64))
    last = len(mags) - 1
    hi = np.minimum(np.searchsorted(mags, a), last)
    lo = np.maximum(hi - 1, 0)
    code = np.where(mags[hi] - a <= a - mags[lo], hi, lo)
    code = np.where(a >= mags[last], last, code) | np.where(np.signbit(v), sign_bit, 0)
    return code.astype(np.uint8)


def test_unmutated_oracle_passes_golden():
    assert _golden_failures() == 0


MUTANTS = {
    "e2m1_ties_away": lambda mp: mp.setattr(Q, "e2m1_encode", lambda v: _ties_away(v, F.E2M1_MAGNITUDES, 8)),
    "e4m3_ties_away": lambda mp: mp.setattr(Q, "e4m3_encode", lambda v: _ties_away(v, F.E4M3_MAGNITUDES, 0x80)),
    "e2m1_drops_sign": lambda mp: mp.setattr(Q, "e2m1_encode", lambda v, f=F.e2m1_encode: f(np.abs(np.asarray(v, np.float32)))),
    "e8m0_floor": lambda mp: mp.setattr(Q, "e8m0_ceil_exponent", lambda s: np.floor(np.log2(np.asarray(s, np.float64))).astype(np.int64)),
    "e8m0_round": lambda mp: mp.setattr(Q, "e8m0_ceil_exponent", lambda s: np.round(np.log2(np.asarray(s, np.float64))).astype(np.int64)),
    "e4m3_decode_bias_8": lambda mp: mp.setattr(Q, "e4m3_decode", lambda c, f=F.e4m3_decode: f(c) / 2.0),
}


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_golden_catches_mutant(name, monkeypatch):
    MUTANTS[name](monkeypatch)
    assert _golden_failures() > 0


def test_golden_catches_nibble_swap(monkeypatch):
    orig = Q.quantize_rank2

    def swapped(fmt, x, tsf=1.0):
        p, s = orig(fmt, x, tsf)
        if fmt != "mxfp8":
            p = ((p >> 4) | (p << 4)).astype(np.uint8)
        return p, s
    monkeypatch.setattr(Q, "quantize_rank2", swapped)
    assert _golden_failures() > 0


def test_golden_catches_dropped_tensor_sf_in_element_scale(monkeypatch):
    # os = 1/ds instead of tensor_sf/ds: visible only where tensor_sf != 1
    orig = Q.nvfp4_element_scale
    monkeypatch.setattr(Q, "nvfp4_element_scale", lambda b, tsf: orig(b, np.float32(1.0)))
    assert _golden_failures() > 0


def test_golden_catches_block_scale_without_tensor_sf(monkeypatch):
    orig = Q.nvfp4_block_scale
    monkeypatch.setattr(Q, "nvfp4_block_scale", lambda a, tsf: orig(a, np.float32(1.0)))
    assert _golden_failures() > 0


def test_golden_catches_mx_qmax_swapped(monkeypatch):
    orig = Q.mx_block_exponent
    monkeypatch.setattr(Q, "mx_block_exponent", lambda a, q: orig(a, 448.0 if q == 6.0 else 6.0))
    assert _golden_failures() > 0


def test_golden_catches_zero_block_scale_one(monkeypatch):
    orig = Q.mx_block_exponent
    monkeypatch.setattr(Q, "mx_block_exponent",
                        lambda a, q: np.where(np.asarray(a) == 0, 0, orig(a, q)))
    assert _golden_failures() > 0


def test_layout_pins_catch_swapped_r32_r4(monkeypatch):
    def wrong(m, s, Kt):
        m = np.asarray(m, dtype=np.int64)
        s = np.asarray(s, dtype=np.int64)
        return (((m // 128) * Kt + s // 4) * 512 + ((m % 128) // 32) * 128
                + (m % 32) * 4 + (s % 4))
    monkeypatch.setattr(L, "offset_5d", wrong)
    sc = np.arange(1, 1 + 128 * 4, dtype=np.int64).reshape(128, 4).astype(np.uint8)
    assert not np.array_equal(L.scales_from_5d_view(L.scales_to_5d(sc), 128, 4), sc)
    assert L.offset_5d(1, 0, 1) != 16
