"""Pins for the oracle's NVFP4 small-M projection (no GPU).

Inputs are written directly as codes and scale bytes, so the expected outputs
follow from the decode tables (pinned in test_oracle_formats.py) by hand or by
a brute-force element loop; asymmetric shapes catch transposed operands, and
distinct per-block scales catch scale-index mistakes.
"""
import numpy as np

from oracle import nvfp4 as Q
from oracle import formats as F


def _pack(el):
    el = np.asarray(el, dtype=np.uint8)
    return (el[:, 0::2] | (el[:, 1::2] << 4)).astype(np.uint8)


def test_identity_weights():
    K = N = 32
    w_el = np.zeros((N, K), np.uint8)
    w_el[np.arange(N), np.arange(K)] = 2                      # E2M1 code 2 = 1.0
    ws = np.full((N, K // 16), 0x38, np.uint8)                 # E4M3 0x38 = 1.0
    rng = np.random.default_rng(0)
    x_el = rng.integers(0, 16, (3, K)).astype(np.uint8)
    xs = np.array([[0x30, 0x40], [0x38, 0x7E], [0x01, 0x08]], np.uint8)
    y, b = Q.gemv(_pack(x_el), xs, np.float32(0.5), _pack(w_el), ws, np.float32(1.0))
    assert np.array_equal(y, Q.dequantize(_pack(x_el), xs, np.float32(0.5)))
    assert np.array_equal(b, np.abs(y))


def test_one_hot_activation_and_nibble_order():
    K, N = 64, 5
    rng = np.random.default_rng(1)
    w_el = rng.integers(0, 16, (N, K)).astype(np.uint8)
    ws = rng.integers(0, 0x7F, (N, K // 16)).astype(np.uint8)
    for kstar in (0, 1, 17, 63):                              # low nibble, high nibble, block 1, last
        x_el = np.zeros((1, K), np.uint8)
        x_el[0, kstar] = 7                                     # 6.0
        xs = np.full((1, K // 16), 0x38, np.uint8)
        y, _ = Q.gemv(_pack(x_el), xs, np.float32(1.0), _pack(w_el), ws, np.float32(2.0))
        want = 6.0 * F.E2M1_VALUES[w_el[:, kstar]] * F.E4M3_VALUES[ws[:, kstar // 16]] * 2.0
        assert np.array_equal(y[0], want)


def test_brute_force_tiny_asymmetric():
    M, N, K = 3, 5, 48
    rng = np.random.default_rng(2)
    x_el = rng.integers(0, 16, (M, K)).astype(np.uint8)
    w_el = rng.integers(0, 16, (N, K)).astype(np.uint8)
    xs = rng.integers(0x20, 0x50, (M, K // 16)).astype(np.uint8)
    ws = rng.integers(0x20, 0x50, (N, K // 16)).astype(np.uint8)
    xg, wg = np.float32(0.75), np.float32(1.5)
    y, b = Q.gemv(_pack(x_el), xs, xg, _pack(w_el), ws, wg)
    for m in range(M):
        for n in range(N):
            acc = 0.0
            mag = 0.0
            for k in range(K):
                xv = F.e2m1_decode_code(int(x_el[m, k])) * F.e4m3_decode_byte(int(xs[m, k // 16])) * 0.75
                wv = F.e2m1_decode_code(int(w_el[n, k])) * F.e4m3_decode_byte(int(ws[n, k // 16])) * 1.5
                acc += xv * wv
                mag += abs(xv * wv)
            assert y[m, n] == acc and b[m, n] == mag


def test_all_equal_blocks_closed_form():
    # every x element 1.5 (code 3) with scale 2.0 (0x40), every w element -0.5 (code 9) with scale 0.25 (0x28)
    M, N, K = 2, 4, 256
    x_el = np.full((M, K), 3, np.uint8)
    w_el = np.full((N, K), 9, np.uint8)
    xs = np.full((M, K // 16), 0x40, np.uint8)
    ws = np.full((N, K // 16), 0x28, np.uint8)
    y, _ = Q.gemv(_pack(x_el), xs, np.float32(1.0), _pack(w_el), ws, np.float32(1.0))
    assert F.e4m3_decode_byte(0x28) == 0.25
    assert np.all(y == K * (1.5 * 2.0) * (-0.5 * 0.25))


def test_quantized_projection_close_to_float():
    # end-to-end sanity: quantize float data and compare with the FP64 float product
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 1024)).astype(np.float32)
    w = (0.02 * rng.standard_normal((64, 1024))).astype(np.float32)
    xq, xs, xg = Q.quantize_f32(x)
    wq, ws, wg = Q.quantize_f32(w)
    y, b = Q.gemv(xq, xs, xg, wq, ws, wg)
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert rel < 0.25
    assert np.all(np.abs(y) <= b + 1e-12)
