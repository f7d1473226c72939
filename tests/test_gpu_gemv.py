"""GPU small-M NVFP4 GEMV vs the oracle.

Tolerance: |y_gpu - y_ref| <= 1e-3 * sum_k |x_k w_k| + 1e-6 per element, with
y_ref and the error scale computed by the oracle in FP64 from the oracle's own
quantization of the same BF16 inputs (the GPU quantizer's codes are first
checked to be identical to the oracle's).
"""
import numpy as np
import pytest
import torch

from oracle import nvfp4 as Q
from nvfp4_w4a4_decode_gemv_gb300 import api, synth
from tests.gpu_util import assert_within, bits, to_np

pytestmark = pytest.mark.gpu


GEMV = {"tc": api.nvfp4_gemv_smallm, "cc": api.nvfp4_gemv_smallm_cudacore}


@pytest.fixture(params=["tc", "cc"])
def gemv(request):
    """Every GEMV test runs on the tensor-core kernel (nvfp4_gemv_smallm, the
    product path) and on the independent CUDA-core kernel (the cross-check)."""
    return GEMV[request.param]


def _run(gemv, M, N, K, seed, w_std=synth.W_STD):
    x = synth.activations(M, K, seed)
    w = synth.weights(N, K, seed + 1000, std=w_std)
    X = api.nvfp4_quantize_act(x.cuda())
    W = api.nvfp4_quantize_act(w.cuda())
    y = to_np(gemv(X, W))
    xq, xs, xg = Q.quantize_bf16(bits(x))
    wq, ws, wg = Q.quantize_bf16(bits(w))
    assert np.array_equal(to_np(X.codes), xq) and np.array_equal(to_np(W.codes), wq)
    assert np.array_equal(to_np(X.scales), xs) and np.array_equal(to_np(W.scales), ws)
    y_ref, bound = Q.gemv(xq, xs, xg, wq, ws, wg)
    assert_within(y, y_ref, bound)
    return X, W, y


def test_single_gemv_512(gemv):
    """M = 1, K = N = 512 (the smallest workload)."""
    _run(gemv, 1, 512, 512, seed=0)


@pytest.mark.parametrize("M", range(1, 9))
def test_all_m_ragged_tiles(gemv, M):
    # N = 1000: 7 full 128-row tiles and a ragged one; K = 768: 3 chunks of 256
    _run(gemv, M, 1000, 768, seed=10 + M)


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (3, 130, 256), (8, 129, 512), (2, 4096, 4096), (8, 3000, 2816),
                                   (5, 384, 25600), (8, 64, 8192)])
def test_shapes(gemv, M, N, K):
    _run(gemv, M, N, K, seed=M * 7 + N)


def test_identity_and_one_hot_weights(gemv):
    K = N = 512
    w = torch.zeros((N, K))
    w[torch.arange(N), torch.arange(K)] = 1.0
    x = synth.activations(4, K, seed=3)
    X = api.nvfp4_quantize_act(x.cuda())
    W = api.nvfp4_quantize_act(w.to(torch.bfloat16).cuda())
    y = to_np(gemv(X, W))
    xq, xs, xg = Q.quantize_bf16(bits(x))
    wq, ws, wg = Q.quantize_bf16(bits(w.to(torch.bfloat16)))
    # identity weights quantize to e2m1 6 * e4m3 448 * (1/2688): exactly 1 in FP64 arithmetic of the oracle
    xh = Q.dequantize(xq, xs, xg)
    wdiag = Q.dequantize(wq, ws, wg).diagonal()
    assert_within(y, xh * wdiag[None, :], np.abs(xh * wdiag[None, :]))


def test_deterministic_and_repeatable(gemv):
    X, W, y1 = _run(gemv, 6, 2000, 2048, seed=5)
    ws = api.GemvWorkspace()
    y2 = to_np(gemv(X, W, workspace=ws.get(6, 2000, 2048)))
    y3 = to_np(gemv(X, W, workspace=ws.get(6, 2000, 2048)))
    assert np.array_equal(y1, y2) and np.array_equal(y2, y3)


@pytest.mark.parametrize("name,K,N", synth.QWEN3_32B + synth.QWEN3_8B + synth.QWEN3_14B)
def test_full_size_sampled_rows(gemv, name, K, N):
    """The benchmark's projection shapes at full size: the GPU quantizes and
    multiplies the whole matrix; the oracle checks 96 sampled output rows (and
    their codes) at every M = 1..8 (each M is its own kernel instance)."""
    w = synth.weights(N, K, seed=777)
    W = api.nvfp4_quantize_act(w.cuda())
    wb = bits(w)
    wf = Q.bf16_bits_to_f32(wb)
    g_ref = Q.global_scale(wf)
    assert to_np(W.global_scale)[0] == g_ref
    rows = np.unique(np.concatenate([np.random.default_rng(N + K).integers(0, N, 94), [0, N - 1]]))
    wq, ws, _ = Q.quantize_f32(wf[rows], g=g_ref)
    assert np.array_equal(to_np(W.codes)[rows], wq) and np.array_equal(to_np(W.scales)[rows], ws)
    for M in range(1, 9):
        x = synth.activations(M, K, seed=900 + M)
        X = api.nvfp4_quantize_act(x.cuda())
        y = to_np(gemv(X, W))
        xq, xs, xg = Q.quantize_bf16(bits(x))
        y_ref, bound = Q.gemv(xq, xs, xg, wq, ws, g_ref)
        assert_within(y[:, rows], y_ref, bound)
