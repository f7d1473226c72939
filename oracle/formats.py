"""E2M1 (FP4) and E4M3 (FP8) element formats, written from their definitions.

NVFP4 stores E2M1 elements with one E4M3 scale per 16-element block and one
FP32 global scale (ReSET reading note, §2.1 "what the NVFP4 format is": E2M1
elements, 16-element blocks with FP8 E4M3 scales, plus an FP32 global scale;
§6.1 setup: E2M1 elements, E4M3 block scales, group size 16).

Encoders are brute force: every finite non-negative value of the format is
listed, the nearest one is taken, a tie between two neighbours goes to the code
whose mantissa LSB (= code LSB) is even, and anything above the largest finite
value saturates to it.  The sign is carried separately by the caller.

Test infrastructure only (see the package docstring).
"""
import numpy as np


def e2m1_decode_code(code: int) -> float:
    """Value of a 4-bit E2M1 code: sign bit 3, exponent bits 2..1 (bias 1),
    mantissa bit 0; exponent 0 is subnormal (0 or 0.5)."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        mag = 0.5 * m
    else:
        mag = 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return -mag if s else mag


def e4m3_decode_byte(b: int) -> float:
    """Value of an E4M3 byte, OCP 'fn' variant: sign bit 7, exponent bits 6..3
    (bias 7), mantissa bits 2..0; exponent 0 is subnormal; 0x7F/0xFF are NaN
    and there is no infinity."""
    s = (b >> 7) & 1
    e = (b >> 3) & 15
    m = b & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        mag = (m / 8.0) * 2.0 ** -6
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


# Decode tables (float64, exact).
E2M1_VALUES = np.array([e2m1_decode_code(c) for c in range(16)], dtype=np.float64)
E4M3_VALUES = np.array([e4m3_decode_byte(b) for b in range(256)], dtype=np.float64)

# Finite non-negative grids, in code order (which is value order).
E2M1_MAG_GRID = E2M1_VALUES[:8]            # codes 0..7: 0, .5, 1, 1.5, 2, 3, 4, 6
E4M3_POS_GRID = E4M3_VALUES[:0x7F]         # codes 0x00..0x7E: 0 .. 448
E2M1_MAX = float(E2M1_MAG_GRID[-1])        # 6
E4M3_MAX = float(E4M3_POS_GRID[-1])        # 448


def _nearest_code_ties_even(t: np.ndarray, grid: np.ndarray, chunk: int = 1 << 16) -> np.ndarray:
    """Index of the grid value nearest to each non-negative t.

    Distances are taken in float64.  t is float32 and the grid values are
    short dyadic rationals, so every distance that can decide the minimum is
    exact in float64 (a far-away candidate may round, but rounding is monotone
    and cannot turn a strictly larger distance into a smaller one).  argmin
    returns the lower index of a tie; the tie then moves to the upper
    neighbour when the lower code is odd, which is ties-to-even on the code.
    Values above the last grid point map to it (saturation): they are clamped
    to it first, because far above the grid every float64 distance rounds to
    the same number and the nearest-value search alone could not tell.
    """
    t = np.asarray(t)
    flat = np.minimum(t.reshape(-1).astype(np.float64), grid[-1])
    out = np.empty(flat.shape, dtype=np.int64)
    last = len(grid) - 1
    for lo in range(0, flat.size, chunk):
        v = flat[lo:lo + chunk]
        dist = np.abs(v[:, None] - grid[None, :])
        idx = np.argmin(dist, axis=1)
        nxt = np.minimum(idx + 1, last)
        rows = np.arange(v.size)
        tie = (idx < last) & (dist[rows, nxt] == dist[rows, idx]) & ((idx & 1) == 1)
        out[lo:lo + chunk] = np.where(tie, idx + 1, idx)
    return out.reshape(t.shape)


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """E2M1 code (uint8, 0..15) of float32 values v: round to nearest, ties to
    even, saturate at 6; the sign bit of the code is the sign bit of v (so a
    negative value that rounds to zero gives the code 0x8)."""
    v = np.asarray(v, dtype=np.float32)
    mag = _nearest_code_ties_even(np.abs(v), E2M1_MAG_GRID)
    sign = np.signbit(v).astype(np.int64) << 3
    return (mag | sign).astype(np.uint8)


def e4m3_encode_nonneg(t: np.ndarray) -> np.ndarray:
    """E4M3 byte of non-negative float32 values t: round to nearest, ties to
    even, saturate at 448 (0x7E)."""
    t = np.asarray(t, dtype=np.float32)
    if np.any(np.signbit(t) & (t != 0)) or np.any(np.isnan(t)):
        raise ValueError("E4M3 block scales are encoded from non-negative, non-NaN values")
    return _nearest_code_ties_even(np.abs(t), E4M3_POS_GRID).astype(np.uint8)


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    return E2M1_VALUES[np.asarray(codes, dtype=np.int64) & 15]


def e4m3_decode(b: np.ndarray) -> np.ndarray:
    return E4M3_VALUES[np.asarray(b, dtype=np.int64) & 255]
