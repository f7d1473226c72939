"""Pins for the oracle's E2M1 / E4M3 codecs (no GPU).

Expected values are hand-derived from the format definitions (E2M1: 1 sign,
2 exponent, 1 mantissa bit; E4M3 'fn': bias 7, max 448, no infinity), or come
from an independent library (ml_dtypes / torch FP8 casts) where it is present.
"""
import math

import numpy as np
import pytest

from oracle import formats as F


def test_e2m1_value_set():
    # The eight FP4 E2M1 magnitudes, written out (not derived from bit fields).
    assert F.E2M1_VALUES[:8].tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert F.E2M1_VALUES[8:].tolist() == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    assert math.copysign(1.0, F.E2M1_VALUES[8]) == -1.0


def test_e2m1_roundtrip_all_codes():
    vals = F.E2M1_VALUES.astype(np.float32)
    assert F.e2m1_encode(vals).tolist() == list(range(16))


@pytest.mark.parametrize("v,code", [
    (0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),   # ties -> even code
    (-0.25, 8), (-0.75, 10), (-1.25, 10), (-1.75, 12), (-2.5, 12), (-3.5, 14), (-5.0, 14),
    (0.2499, 0), (0.2501, 1), (0.7499, 1), (0.7501, 2), (4.99, 6), (5.01, 7),
    (6.0, 7), (6.49, 7), (6.5, 7), (7.0, 7), (100.0, 7), (1e30, 7),             # saturation
    (-6.5, 15), (-1e30, 15),
    (-0.1, 8), (-0.0, 8), (0.0, 0), (1e-30, 0),                                  # sign kept at zero
])
def test_e2m1_hand_worked(v, code):
    assert int(F.e2m1_encode(np.float32(v))) == code


def test_e2m1_against_library():
    md = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(0)
    v = np.concatenate([
        np.arange(-8 * 64, 8 * 64 + 1, dtype=np.float32) / 64,   # all ties and grid points
        rng.uniform(-9, 9, 20000).astype(np.float32),
        rng.standard_normal(20000).astype(np.float32) * 1e-3,
    ]).astype(np.float32)
    lib = v.astype(md.float4_e2m1fn).view(np.uint8) & 15
    assert np.array_equal(F.e2m1_encode(v), lib)


@pytest.mark.parametrize("b,val", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
    (0x38, 1.0), (0x39, 1.125), (0x3F, 1.875), (0x40, 2.0), (0x76, 224.0), (0x7E, 448.0),
    (0x80, -0.0), (0xB8, -1.0), (0xFE, -448.0),
])
def test_e4m3_known_values(b, val):
    got = F.e4m3_decode_byte(b)
    assert got == val and math.copysign(1.0, got) == math.copysign(1.0, val)


def test_e4m3_nan_and_order():
    assert math.isnan(F.e4m3_decode_byte(0x7F)) and math.isnan(F.e4m3_decode_byte(0xFF))
    pos = F.E4M3_POS_GRID
    assert len(pos) == 127 and np.all(np.diff(pos) > 0)
    assert F.E4M3_MAX == 448.0


def test_e4m3_decode_against_libraries():
    allb = np.arange(256, dtype=np.uint8)
    mine = F.e4m3_decode(allb)
    torch = pytest.importorskip("torch")
    tv = torch.from_numpy(allb.copy()).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    assert np.array_equal(np.isnan(mine), np.isnan(tv))
    ok = ~np.isnan(mine)
    assert np.array_equal(mine[ok], tv[ok])
    md = pytest.importorskip("ml_dtypes")
    lv = allb.view(md.float8_e4m3fn).astype(np.float64)
    assert np.array_equal(mine[ok], lv[ok])


@pytest.mark.parametrize("t,b", [
    (448.0, 0x7E), (460.0, 0x7E), (464.0, 0x7E), (500.0, 0x7E), (1e9, 0x7E),   # saturation
    (2.0 ** -9, 0x01), (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02),              # subnormal ties
    (1.0625, 0x38), (1.1875, 0x3A), (1.0624, 0x38), (1.0626, 0x39),            # normal ties
    (224.0, 0x76), (240.0, 0x77), (256.0, 0x78), (0.0, 0x00),
])
def test_e4m3_encode_hand_worked(t, b):
    assert int(F.e4m3_encode_nonneg(np.float32(t))) == b


def test_e4m3_encode_against_libraries():
    rng = np.random.default_rng(1)
    t = np.concatenate([
        F.E4M3_POS_GRID.astype(np.float32),
        ((F.E4M3_POS_GRID[:-1] + F.E4M3_POS_GRID[1:]) / 2).astype(np.float32),   # every tie point
        np.exp(rng.uniform(np.log(1e-5), np.log(460.0), 30000)).astype(np.float32),
    ]).astype(np.float32)
    mine = F.e4m3_encode_nonneg(t)
    torch = pytest.importorskip("torch")
    tb = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, tb)
    md = pytest.importorskip("ml_dtypes")
    assert np.array_equal(mine, t.astype(md.float8_e4m3fn).view(np.uint8))


def test_e4m3_rejects_negative():
    with pytest.raises(ValueError):
        F.e4m3_encode_nonneg(np.float32(-1.0))
