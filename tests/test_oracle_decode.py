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


def test_rms_norm_closed_forms():
    # a row [3, 4]: mean square 12.5, so the values are 3/sqrt(12.5), 4/sqrt(12.5)
    r = D.rms_norm(np.array([[3.0, 4.0]]), 0.0)
    assert np.allclose(r, [[3 / np.sqrt(12.5), 4 / np.sqrt(12.5)]], rtol=0, atol=1e-15)
    # a constant row c with eps: c / sqrt(c^2 + eps); rows are independent
    r = D.rms_norm(np.array([[2.0] * 8, [-0.5] * 8]), 0.25)
    assert np.allclose(r[0], 2 / np.sqrt(4.25)) and np.allclose(r[1], -0.5 / np.sqrt(0.5))
    # scale invariance at eps = 0, and the output has mean square 1
    x = np.random.default_rng(0).standard_normal((3, 64))
    assert np.allclose(D.rms_norm(x, 0.0), D.rms_norm(7.5 * x, 0.0))
    assert np.allclose(np.mean(D.rms_norm(x, 0.0) ** 2, axis=1), 1.0)
    # a zero row stays zero when eps > 0
    assert np.all(D.rms_norm(np.zeros((1, 16)), 1e-6) == 0)
