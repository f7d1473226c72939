"""GPU GEMV on packed weights (nvfp4_pack_weights + nvfp4_gemv_smallm_packed).

The packed image is checked byte for byte against the layout nvfp4.h defines
(written out here in numpy from that definition); the packed GEMV against the
oracle with the GEMV tolerance |y - y_ref| <= 1e-3 * sum_k |x_k w_k| + 1e-6,
and bit for bit against the tensor-core GEMV on the row-major weights.
"""
import numpy as np
import pytest
import torch

from oracle import nvfp4 as Q
from nvfp4_w4a4_decode_gemv_gb300 import api, synth
from tests.gpu_util import assert_within, bits, to_np

pytestmark = pytest.mark.gpu


def _layout(wq, ws, N, K):
    """The packed layout of nvfp4.h, from its definition."""
    T, C = (N + 127) // 128, K // 256
    out = np.zeros((T, C, 18432), np.uint8)
    for t in range(T):
        for c in range(C):
            for r in range(128):
                n = 128 * t + r
                if n >= N:
                    continue
                for j in range(8):
                    d = r * 128 + (j ^ (r % 8)) * 16
                    out[t, c, d:d + 16] = wq[n, 128 * c + 16 * j: 128 * c + 16 * j + 16]
                out[t, c, 16384 + 16 * r: 16384 + 16 * r + 16] = ws[n, 16 * c: 16 * c + 16]
    return out.reshape(-1)


@pytest.mark.parametrize("N,K", [(1000, 768), (128, 256), (1, 512)])
def test_pack_layout(N, K):
    w = synth.weights(N, K, seed=N + K)
    W = api.nvfp4_quantize_act(w.cuda())
    P = api.nvfp4_pack_weights(W)
    assert P.packed.numel() == api.nvfp4_packed_weight_bytes(N, K) == ((N + 127) // 128) * (K // 256) * 18432
    assert np.array_equal(to_np(P.packed), _layout(to_np(W.codes), to_np(W.scales), N, K))


def _run(M, N, K, seed):
    x = synth.activations(M, K, seed)
    w = synth.weights(N, K, seed + 1000)
    X = api.nvfp4_quantize_act(x.cuda())
    W = api.nvfp4_quantize_act(w.cuda())
    P = api.nvfp4_pack_weights(W)
    y = to_np(api.nvfp4_gemv_smallm_packed(X, P))
    xq, xs, xg = Q.quantize_bf16(bits(x))
    wq, ws, wg = Q.quantize_bf16(bits(w))
    assert np.array_equal(to_np(W.codes), wq) and np.array_equal(to_np(W.scales), ws)
    y_ref, bound = Q.gemv(xq, xs, xg, wq, ws, wg)
    assert_within(y, y_ref, bound)
    y_rowmajor = to_np(api.nvfp4_gemv_smallm(X, W))
    assert np.array_equal(y.view(np.uint32), y_rowmajor.view(np.uint32))


@pytest.mark.parametrize("M", range(1, 9))
def test_all_m_ragged(M):
    _run(M, 1000, 768, seed=20 + M)


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (3, 130, 256), (8, 129, 512), (2, 4096, 4096), (8, 3000, 2816),
                                   (5, 384, 25600), (8, 64, 8192)])
def test_shapes(M, N, K):
    _run(M, N, K, seed=M * 11 + N)


def test_repeatable_across_workspaces():
    M, N, K = 7, 2000, 2048
    X = api.nvfp4_quantize_act(synth.activations(M, K, 4).cuda())
    P = api.nvfp4_pack_weights(api.nvfp4_quantize_act(synth.weights(N, K, 5).cuda()))
    ys = [to_np(api.nvfp4_gemv_smallm_packed(X, P, workspace=api.GemvWorkspace().get(M, N, K))) for _ in range(3)]
    assert all(np.array_equal(ys[0], y) for y in ys[1:])


@pytest.mark.parametrize("name,K,N", synth.QWEN3_32B)
def test_full_size_sampled_rows(name, K, N):
    """Full-size Qwen3-32B projections, packed: 96 sampled output rows checked by the oracle at every M = 1..8."""
    w = synth.weights(N, K, seed=778)
    W = api.nvfp4_quantize_act(w.cuda())
    P = api.nvfp4_pack_weights(W)
    wf = Q.bf16_bits_to_f32(bits(w))
    g_ref = Q.global_scale(wf)
    rows = np.unique(np.concatenate([np.random.default_rng(N * 3 + K).integers(0, N, 94), [0, N - 1]]))
    wq, ws, _ = Q.quantize_f32(wf[rows], g=g_ref)
    del W
    for M in range(1, 9):
        x = synth.activations(M, K, seed=910 + M)
        X = api.nvfp4_quantize_act(x.cuda())
        y = to_np(api.nvfp4_gemv_smallm_packed(X, P))
        xq, xs, xg = Q.quantize_bf16(bits(x))
        y_ref, bound = Q.gemv(xq, xs, xg, wq, ws, g_ref)
        assert_within(y[:, rows], y_ref, bound)


def test_shapes_back_to_back_on_one_workspace():
    """Calls of different shapes queued back to back on one workspace (each may
    start before the previous one ends) give the bits of isolated calls."""
    shapes = [(8, 10240, 5120), (1, 1000, 768), (4, 5120, 8192), (8, 51200, 512), (2, 384, 25600), (1, 129, 256)]
    ops = []
    for i, (M, N, K) in enumerate(shapes):
        X = api.nvfp4_quantize_act(synth.activations(M, K, 60 + i).cuda())
        P = api.nvfp4_pack_weights(api.nvfp4_quantize_act(synth.weights(N, K, 70 + i).cuda()))
        ref = to_np(api.nvfp4_gemv_smallm_packed(X, P, workspace=api.GemvWorkspace().get(M, N, K)))
        ops.append((X, P, ref))
    need = max(api.nvfp4_gemv_workspace_bytes(M, N, K) for M, N, K in shapes)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for rep in range(3):
        ys = [api.nvfp4_gemv_smallm_packed(X, P, workspace=ws) for X, P, _ in ops]
        for (X, P, ref), y in zip(ops, ys):
            assert np.array_equal(to_np(y).view(np.uint32), ref.view(np.uint32))
