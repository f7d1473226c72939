"""The prefill-sized NVFP4 GEMM (nvfp4_gemm_packed, M up to 128) vs the oracle.

Tolerance as for the GEMV: |y - y_ref| <= 1e-3 * sum_k |x_k w_k| + 1e-6 per
element, y_ref in FP64 from the oracle's own quantization of the same BF16
inputs (whose codes the GPU quantizer reproduces bit for bit).  Also: the
full-size Qwen3-32B projections at M = 128 on sampled output rows, repeat and
back-to-back calls bit for bit on one workspace, agreement with the GEMV at
M <= 8, output canaries and the fix-up's bounded wait made to run out.
"""
import numpy as np
import pytest
import torch

from oracle import nvfp4 as Q
from nvfp4_w4a4_decode_gemv_gb300 import api, synth
from nvfp4_w4a4_decode_gemv_gb300._lib import lib
from tests.gpu_util import Guarded, assert_within, bits, to_np

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed):
    x = synth.activations(M, K, seed)
    w = synth.weights(N, K, seed + 1000)
    X = api.nvfp4_quantize_act(x.cuda())
    P = api.nvfp4_pack_weights(api.nvfp4_quantize_act(w.cuda()))
    return x, w, X, P


def _oracle(x, w):
    xq, xs, xg = Q.quantize_bf16(bits(x))
    wq, ws, wg = Q.quantize_bf16(bits(w))
    return Q.gemv(xq, xs, xg, wq, ws, wg)


@pytest.mark.parametrize("M", [1, 2, 9, 16, 17, 33, 64, 100, 127, 128])
def test_gemm_every_m_class_ragged(M):
    x, w, X, P = _operands(M, 1000, 768, seed=50 + M)
    y = to_np(api.nvfp4_gemm_packed(X, P))
    y_ref, bound = _oracle(x, w)
    assert_within(y, y_ref, bound)
    assert api.device_status() == 0


@pytest.mark.parametrize("M", [1, 17, 100, 128])
def test_gemm_split_tiles_ragged_m(M):
    """N = 300 (3 tiles), K = 25600: every tile split across 50 CTAs, their
    partial sums merged by the tile's first CTA, for ragged token counts."""
    x, w, X, P = _operands(M, 300, 25600, seed=60 + M)
    y = to_np(api.nvfp4_gemm_packed(X, P))
    y_ref, bound = _oracle(x, w)
    assert_within(y, y_ref, bound)
    assert api.device_status() == 0


@pytest.mark.parametrize("M,N,K", [(128, 1, 256), (128, 129, 256), (96, 3000, 2816), (128, 384, 25600),
                                   (40, 64, 8192), (128, 4096, 4096)])
def test_gemm_shapes(M, N, K):
    x, w, X, P = _operands(M, N, K, seed=M + N + K)
    y = to_np(api.nvfp4_gemm_packed(X, P))
    y_ref, bound = _oracle(x, w)
    assert_within(y, y_ref, bound)


@pytest.mark.parametrize("name,K,N", synth.QWEN3_32B)
def test_gemm_full_size_m128(name, K, N):
    """The Qwen3-32B projections at M = 128: 96 sampled output rows against
    the oracle."""
    M = 128
    w = synth.weights(N, K, seed=781)
    P = api.nvfp4_pack_weights(api.nvfp4_quantize_act(w.cuda()))
    wf = Q.bf16_bits_to_f32(bits(w))
    g_ref = Q.global_scale(wf)
    rows = np.unique(np.concatenate([np.random.default_rng(N * 7 + K).integers(0, N, 94), [0, N - 1]]))
    wq, ws, _ = Q.quantize_f32(wf[rows], g=g_ref)
    x = synth.activations(M, K, seed=940)
    X = api.nvfp4_quantize_act(x.cuda())
    y = to_np(api.nvfp4_gemm_packed(X, P))
    xq, xs, xg = Q.quantize_bf16(bits(x))
    assert np.array_equal(to_np(X.codes), xq) and np.array_equal(to_np(X.scales), xs)
    y_ref, bound = Q.gemv(xq, xs, xg, wq, ws, g_ref)
    assert_within(y[:, rows], y_ref, bound)
    assert api.device_status() == 0


def test_gemm_matches_gemv_at_small_m():
    for M in (1, 5, 8):
        x, w, X, P = _operands(M, 2000, 2048, seed=70 + M)
        y1 = to_np(api.nvfp4_gemm_packed(X, P))
        y2 = to_np(api.nvfp4_gemv_smallm_packed(X, P))
        _, bound = _oracle(x, w)
        assert np.all(np.abs(y1.astype(np.float64) - y2) <= 2e-3 * bound + 2e-6)


def test_gemm_repeatable_and_back_to_back():
    shapes = [(128, 10240, 5120), (7, 1000, 768), (128, 5120, 8192), (64, 51200, 512), (128, 384, 25600),
              (1, 129, 256)]
    ops = []
    for i, (M, N, K) in enumerate(shapes):
        _, _, X, P = _operands(M, N, K, seed=200 + i)
        ws0 = torch.zeros(api.nvfp4_gemm_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
        ops.append((X, P, to_np(api.nvfp4_gemm_packed(X, P, workspace=ws0))))
    need = max(api.nvfp4_gemm_workspace_bytes(M, N, K) for M, N, K in shapes)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for rep in range(3):
        ys = [api.nvfp4_gemm_packed(X, P, workspace=ws) for X, P, _ in ops]
        for (X, P, ref), y in zip(ops, ys):
            assert np.array_equal(to_np(y).view(np.uint32), ref.view(np.uint32)), rep
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(ws)) == 0
    assert api.device_status() == 0


@pytest.mark.parametrize("M,N,K", [(128, 1, 256), (33, 129, 768), (128, 1000, 2816)])
def test_gemm_canaries(M, N, K):
    x, w, X, P = _operands(M, N, K, seed=300 + M)
    y = Guarded((M, N), torch.float32)
    api.nvfp4_gemm_packed(X, P, y=y.t)
    y.check("y")
    y_ref, bound = _oracle(x, w)
    assert_within(to_np(y.t), y_ref, bound)


@pytest.mark.parametrize("M,N,K", [(33, 4999, 25600), (16, 5120, 25600)])
def test_gemm_cluster_plan_canaries(M, N, K):
    """40 tiles of 100 steps: each tile on a cluster of three CTAs whose
    partial sums rank 0 adds over distributed shared memory; y inside guard
    bands (N = 4999: scalar stores; N = 5120: the staged bulk stores)."""
    x, w, X, P = _operands(M, N, K, seed=500 + M)
    y = Guarded((M, N), torch.float32)
    api.nvfp4_gemm_packed(X, P, y=y.t)
    y.check("y")
    y_ref, bound = _oracle(x, w)
    assert_within(to_np(y.t), y_ref, bound)
    assert api.device_status() == 0


def test_gemm_fixup_wait_runs_out_and_is_reported():
    M, N, K = 16, 300, 25600         # 300 units, 150 CTAs of two: every tile split across 50 CTAs
    x, w, X, P = _operands(M, N, K, seed=400)
    ws = torch.zeros(api.nvfp4_gemm_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    assert api.device_status() == 0
    L = lib()
    L.nvfp4_test_gemv_fault(1 << 10, 1)
    try:
        api.nvfp4_gemm_packed(X, P, workspace=ws)
        torch.cuda.synchronize()
    finally:
        L.nvfp4_test_gemv_fault(0, 0)
    assert int(torch.count_nonzero(ws)) == 0
    assert api.device_status() == api.DEVERR_FLAG_TIMEOUT
    y = to_np(api.nvfp4_gemm_packed(X, P, workspace=ws))
    y_ref, bound = _oracle(x, w)
    assert_within(y, y_ref, bound)
    assert api.device_status() == 0
