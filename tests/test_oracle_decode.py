"""Pins for the oracle's decode-step glue: SiLU * mul and the BF16 lm_head GEMV (no GPU)."""
import math

import numpy as np
import pytest

from oracle import decode as D
from oracle import nvfp4 as Q


def test_silu_known_values():
    assert D.silu(np.array([0.0]))[0] == 0.0
    assert D.silu(np.array([1.0]))[0] == pytest.approx(1 / (1 + math.exp(-1)), rel=1e-15)
    assert D.silu(np.array([-2.0]))[0] == pytest.approx(-2 / (1 + math.exp(2)), rel=1e-15)
    assert D.silu(np.array([40.0]))[0] == pytest.approx(40.0, rel=1e-15)
    assert abs(D.silu(np.array([-40.0]))[0]) < 1e-15


def test_silu_mul_halves():
    gu = np.array([[1.0, 2.0, 10.0, 20.0], [0.0, -1.0, 3.0, 4.0]])
    out = D.silu_mul(gu)                    # gate = first half, up = second half
    want = np.array([[D.silu(np.array([1.0]))[0] * 10, D.silu(np.array([2.0]))[0] * 20],
                     [0.0, D.silu(np.array([-1.0]))[0] * 4]])
    assert np.array_equal(out, want)


def test_bf16_gemv_hand():
    x = Q.f32_to_bf16_bits(np.array([[1.0, -2.0, 0.5]], np.float32))
    w = Q.f32_to_bf16_bits(np.array([[1.0, 1.0, 1.0], [0.25, 0.5, -4.0]], np.float32))
    y, b = D.bf16_gemv(x, w)
    assert y.tolist() == [[-0.5, -2.75]] and b.tolist() == [[3.5, 3.25]]


def test_to_bf16_rounds_through_fp32():
    # 1 + 2^-8 + 2^-30 rounds to FP32 1 + 2^-8 (a BF16 tie) and then to 1.0
    v = 1 + 2.0 ** -8 + 2.0 ** -30
    assert D.to_bf16_bits(np.array([v]))[0] == 0x3F80


def test_table4_fixture_shapes():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "table4_m1_gemv_shapes.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    assert len(rows) == 12
    for model, layer, N, K, ours, theirs in rows:
        assert int(K) % 256 == 0 and int(N) % 256 == 0
        assert 1.5 < float(theirs) / float(ours) < 2.6
