"""NVFP4 quantize / dequantize / small-M projection, plain and slow.

Format (ReSET reading note, §2.1 and §6.1 setup): E2M1 elements, one E4M3
scale per 16 consecutive elements along K, one FP32 global scale per tensor.
Layout: codes[r, j] holds element 2j in the low nibble and 2j+1 in the high
nibble; scales[r, b] is the scale of elements 16b..16b+15 of row r (row-major,
not interleaved -- the pages' pipeline feeds a non-interleaved scale layout,
reading note §5.3).

Quantize recipe, FP32 with one rounding per operation, in this order:
  amax = max |x| over the whole tensor        (exact)
  g    = amax / 2688                          (448 * 6: largest E4M3 * largest E2M1)
  per row r, block b:  bm = max |x| in the block,  d = 6 * g,  t = bm / d,
                       s = E4M3(t)  (nearest, ties to even, saturating)
  per element:         S = dec(s) * g,  v = x / S,  c = E2M1(v)
Readings where the recipe leaves a case open (each pinned by a test):
  * a negative value that rounds to magnitude 0 keeps its sign: code 0x8;
  * when S == 0 (all-zero block, a scale that underflows to 0, or an all-zero
    tensor) the magnitude is 0 and the code is the sign bit of x alone;
  * non-finite inputs are outside the contract and raise here.
Dequantization multiplies: x_hat = E2M1(c) * E4M3(s) * g, exact in FP64.

The projection is Y[m, n] = sum_k x_hat[m, k] * w_hat[n, k] in FP64 (ReSET
project page, "Core contribution": Y = X W computed at small M).  The error
scale used by the parity tests is B[m, n] = sum_k |x_hat[m, k] * w_hat[n, k]|.

Test infrastructure only (see the package docstring).
"""
import numpy as np

from .formats import e2m1_encode, e4m3_encode_nonneg, e2m1_decode, e4m3_decode

BLOCK = 16
GLOBAL_DIVISOR = np.float32(2688.0)   # 448 * 6, exact in FP32
SIX = np.float32(6.0)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns (uint16) to float32 values; exact."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def global_scale(x: np.ndarray) -> np.float32:
    """g = amax / 2688 over the whole float32 tensor x."""
    if x.size == 0:
        return np.float32(0.0)
    amax = np.float32(np.max(np.abs(x)))
    return np.float32(amax / GLOBAL_DIVISOR)


def quantize_f32(x: np.ndarray, g: np.float32 | None = None):
    """Quantize float32 x[rows, K] (K % 16 == 0).

    Returns (codes uint8 [rows, K/2], scales uint8 [rows, K/16], g float32).
    g defaults to the recipe's amax / 2688 over x.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim != 2 or x.shape[1] % BLOCK != 0:
        raise ValueError("x must be [rows, K] with K a multiple of 16")
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite input is outside the NVFP4 quantize contract")
    rows, K = x.shape
    nb = K // BLOCK
    if g is None:
        g = global_scale(x)
    g = np.float32(g)

    absx = np.abs(x)
    bm = absx.reshape(rows, nb, BLOCK).max(axis=2) if x.size else np.zeros((rows, nb), np.float32)
    d = np.float32(SIX * g)
    if d == 0:
        t = np.zeros_like(bm)
    else:
        t = (bm / d).astype(np.float32)
    s = e4m3_encode_nonneg(t)                                   # [rows, nb]

    S = (e4m3_decode(s).astype(np.float32) * g).astype(np.float32)
    S_el = np.repeat(S, BLOCK, axis=1)                          # [rows, K]
    nz = S_el != 0
    v = np.zeros_like(x)
    v[nz] = x[nz] / S_el[nz]                                    # float32 division
    c = e2m1_encode(v)                                          # magnitude of v, sign of v
    sign_only = (np.signbit(x).astype(np.uint8) << 3)
    c = np.where(nz, (c & 7) | sign_only, sign_only).astype(np.uint8)

    codes = (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    return codes, s, g


def quantize_bf16(bits: np.ndarray, g: np.float32 | None = None):
    """Quantize a BF16 tensor given as uint16 bit patterns [rows, K]."""
    return quantize_f32(bf16_bits_to_f32(bits), g)


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    """codes uint8 [rows, K/2] -> element codes uint8 [rows, K] (low nibble first)."""
    codes = np.asarray(codes, dtype=np.uint8)
    out = np.empty((codes.shape[0], codes.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = codes & 15
    out[:, 1::2] = codes >> 4
    return out


def dequantize(codes: np.ndarray, scales: np.ndarray, g) -> np.ndarray:
    """x_hat = E2M1(c) * E4M3(s) * g in FP64 (exact)."""
    el = e2m1_decode(unpack_codes(codes))                        # [rows, K] f64
    sc = np.repeat(e4m3_decode(scales), BLOCK, axis=1)           # [rows, K] f64
    return el * sc * np.float64(np.float32(g))


def gemv(xq, xs, xg, wq, ws, wg):
    """Y[m, n] = sum_k x_hat[m, k] w_hat[n, k] and its error scale, both FP64 [M, N]."""
    xh = dequantize(xq, xs, xg)
    wh = dequantize(wq, ws, wg)
    return xh @ wh.T, np.abs(xh) @ np.abs(wh).T


def gemv_tolerance(bound: np.ndarray) -> np.ndarray:
    """Allowed |y_gpu - y_ref| per element: 1e-3 * sum_k |x_k w_k| + 1e-6."""
    return 1e-3 * bound + 1e-6
