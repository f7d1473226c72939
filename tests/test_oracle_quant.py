"""Pins for the oracle's NVFP4 quantize recipe (no GPU).

The worked example is built so that every FP32 step of the recipe is exact
(tensor amax 2688 = 448 * 6 gives g = 1), so the expected scales and codes
follow by hand from the format tables and the tie rules.
"""
import numpy as np
import pytest

from oracle import nvfp4 as Q
from oracle import formats as F


def _worked_example():
    x = np.zeros((2, 48), dtype=np.float32)
    # row 0, block 0: amax 2688 -> g = 1, d = 6, t = 448 -> s = 0x7E, S = 448
    x[0, 0:16] = 448 * np.array([0, .25, .5, .75, 1, 1.25, 1.5, 1.75, 2, 2.5, 3, 3.5, 4, 5, 6, -6])
    # row 0, block 1: bm = 1344 -> t = 224 -> s = 0x76, S = 224
    x[0, 16:32] = 224 * np.array([6, -6, 3, -3, 1.5, -1.5, .5, -.5, .25, -.25, 2.5, -2.5, 0, -0.0, 4, -4])
    # row 0, block 2: bm = 6.375 -> t = 1.0625, a tie between 1.0 and 1.125 -> 1.0 (0x38), S = 1
    x[0, 32:36] = [6.375, 1.0, -1.25, 0.75]
    # row 1, block 0: all zero with one -0.0 -> s = 0, S = 0: codes are the sign bits
    x[1, 1] = -0.0
    # row 1, block 1: bm = 6 * 2^-10 -> t = 2^-10, a tie between 0 and 2^-9 -> s = 0, S = 0
    x[1, 16:19] = [6 * 2.0 ** -10, -6 * 2.0 ** -10, 2.0 ** -10]
    # row 1, block 2: bm = 18 * 2^-9 -> t = 3 * 2^-9 (E4M3 subnormal 0x03), S = 3 * 2^-9
    S = 3 * 2.0 ** -9
    x[1, 32:36] = [6 * S, 1 * S, -0.5 * S, 2 * S]
    return x


def test_worked_example_codes_and_scales():
    x = _worked_example()
    bits = Q.f32_to_bf16_bits(x)
    assert np.array_equal(Q.bf16_bits_to_f32(bits), x), "example values must be exact in BF16"
    codes, scales, g = Q.quantize_bf16(bits)
    assert g == np.float32(1.0)
    assert scales.tolist() == [[0x7E, 0x76, 0x38], [0x00, 0x00, 0x03]]
    el = Q.unpack_codes(codes)
    assert el[0, 0:16].tolist() == [0, 0, 1, 2, 2, 2, 3, 4, 4, 4, 5, 6, 6, 6, 7, 15]
    assert el[0, 16:32].tolist() == [7, 15, 5, 13, 3, 11, 1, 9, 0, 8, 4, 12, 0, 8, 6, 14]
    assert el[0, 32:48].tolist() == [7, 2, 10, 2] + [0] * 12
    assert el[1, 0:16].tolist() == [0, 8] + [0] * 14
    assert el[1, 16:32].tolist() == [0, 8, 0] + [0] * 13
    assert el[1, 32:48].tolist() == [7, 2, 9, 4] + [0] * 12
    # packing: element 2j in the low nibble, 2j+1 in the high nibble
    assert codes[0, 0:8].tolist() == [0x00, 0x21, 0x22, 0x43, 0x44, 0x65, 0x66, 0xF7]


def test_worked_example_dequant():
    x = _worked_example()
    codes, scales, g = Q.quantize_bf16(Q.f32_to_bf16_bits(x))
    xh = Q.dequantize(codes, scales, g)
    # block 0 of row 0: 448 * E2M1(code)
    want = 448 * np.array([0, 0, .5, 1, 1, 1, 1.5, 2, 2, 2, 3, 4, 4, 4, 6, -6])
    assert np.array_equal(xh[0, :16], want)
    assert np.array_equal(xh[0, 32:36], [6.0, 1.0, -1.0, 1.0])
    assert np.all(xh[1, :32] == 0)


def test_zero_tensor():
    codes, scales, g = Q.quantize_f32(np.zeros((3, 32), np.float32))
    assert g == 0 and not codes.any() and not scales.any()
    x = np.zeros((1, 16), np.float32)
    x[0, 3] = -0.0
    codes, _, _ = Q.quantize_f32(x)
    assert Q.unpack_codes(codes)[0].tolist() == [0, 0, 0, 8] + [0] * 12


def test_empty_and_bad_shapes():
    codes, scales, g = Q.quantize_f32(np.zeros((0, 64), np.float32))
    assert codes.shape == (0, 32) and scales.shape == (0, 4) and g == 0
    with pytest.raises(ValueError):
        Q.quantize_f32(np.zeros((2, 24), np.float32))
    with pytest.raises(ValueError):
        Q.quantize_f32(np.array([[np.inf] + [0] * 15], np.float32))


def _random_bf16(rows, K, seed, outliers=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, K)).astype(np.float32)
    if outliers:
        ch = rng.permutation(K)[: max(1, K // 100)]
        x[:, ch] *= 20
    return Q.f32_to_bf16_bits(x)


def test_invariants_random():
    bits = _random_bf16(8, 4096, 3)
    x = Q.bf16_bits_to_f32(bits).astype(np.float64)
    codes, scales, g = Q.quantize_bf16(bits)
    # the block holding the tensor amax gets t ~ 448 -> the largest scale 0x7E
    assert scales.max() == 0x7E
    assert g == np.float32(np.float32(np.abs(x).max()) / np.float32(2688))
    xh = Q.dequantize(codes, scales, g)
    S = np.repeat(F.e4m3_decode(scales) * np.float64(g), 16, axis=1)
    # nearest-value rounding: error at most one E2M1 step (2 near the top) times half, times S,
    # plus saturation slack above 6 (t rounds to at most 1/16 below bm / 6g)
    assert np.all(np.abs(x - xh) <= S * 1.0 + np.abs(x) * 0.07)
    assert np.all((np.sign(xh) == np.sign(x)) | (xh == 0))
    # relative reconstruction error of the whole tensor stays in the NVFP4 range
    rel = np.linalg.norm(x - xh) / np.linalg.norm(x)
    assert 0.02 < rel < 0.2


def test_recipe_against_library_rounding():
    """The same recipe with an independent library doing both roundings."""
    md = pytest.importorskip("ml_dtypes")
    bits = _random_bf16(4, 2048, 5)
    x = Q.bf16_bits_to_f32(bits)
    codes, scales, g = Q.quantize_bf16(bits)
    amax = np.float32(np.abs(x).max())
    g2 = np.float32(amax / np.float32(2688))
    bm = np.abs(x).reshape(4, -1, 16).max(axis=2)
    t = (bm / np.float32(6 * g2)).astype(np.float32)
    s2 = t.astype(md.float8_e4m3fn)
    S = (s2.astype(np.float32) * g2).astype(np.float32)
    v = (x / np.repeat(S, 16, axis=1)).astype(np.float32)
    c2 = v.astype(md.float4_e2m1fn).view(np.uint8) & 15
    assert g == g2
    assert np.array_equal(scales, s2.view(np.uint8))
    assert np.array_equal(Q.unpack_codes(codes), c2)


def test_bf16_rounding_against_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(50000).astype(np.float32),
                        np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -1 - 2.0 ** -8], np.float32)])
    mine = Q.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)
    # hand ties: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> 1.0 (even)
    assert mine[-3] == 0x3F80 and mine[-2] == 0x3F82 and mine[-1] == 0xBF80
