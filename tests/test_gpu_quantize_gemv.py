"""The quantizer and the packed GEMV as one call (nvfp4_quantize_gemv_packed).

Its result must be the bits of nvfp4_quantize_act followed by
nvfp4_gemv_smallm_packed on the same inputs (whether the library runs it as
one launch or two), its global scale the quantizer's, and y within the GEMV
tolerance |y - y_ref| <= 1e-3 * sum_k |x_k w_k| + 1e-6 of the oracle's
quantize-then-multiply.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from oracle import nvfp4 as Q
from nvfp4_w4a4_decode_gemv_gb300 import api, synth
from tests.gpu_util import assert_within, bits, to_np

pytestmark = pytest.mark.gpu


def _two_calls(x, P, M, N, K):
    X = api.nvfp4_quantize_act(x)
    y = api.nvfp4_gemv_smallm_packed(X, P, workspace=api.GemvWorkspace().get(M, N, K))
    return to_np(y), to_np(X.global_scale)


def _check(M, N, K, seed, oracle=False, x=None):
    x = (x if x is not None else synth.activations(M, K, seed)).cuda()
    w = synth.weights(N, K, seed + 500)
    W = api.nvfp4_quantize_act(w.cuda())
    P = api.nvfp4_pack_weights(W)
    xg = torch.empty(1, dtype=torch.float32, device="cuda")
    y = to_np(api.nvfp4_quantize_gemv_packed(x, P, xg_out=xg))
    y2, g2 = _two_calls(x, P, M, N, K)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32)), (M, N, K)
    assert to_np(xg).view(np.uint32)[0] == g2.view(np.uint32)[0]
    if oracle:
        xq, xs, xgr = Q.quantize_bf16(bits(x.cpu()))
        wq, ws, wg = Q.quantize_bf16(bits(w))
        y_ref, bound = Q.gemv(xq, xs, xgr, wq, ws, wg)
        assert_within(y, y_ref, bound)
    return y


@pytest.mark.parametrize("M", range(1, 9))
def test_all_m_ragged_against_oracle(M):
    """Ragged N (8 tiles, the last one partial), three K chunks: split tiles and whole ones."""
    _check(M, 1000, 768, seed=40 + M, oracle=True)


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (3, 130, 256), (2, 129, 512), (2, 4096, 4096), (3, 3000, 2816),
                                   (1, 64, 8192), (3, 51200, 256), (1, 300, 25600), (8, 3000, 2816), (5, 51200, 256)])
def test_shapes(M, N, K):
    """One launch for M <= 3 (and M * K <= 65536), two above."""
    _check(M, N, K, seed=M * 13 + N, oracle=N * K <= 3000 * 2816)


@pytest.mark.parametrize("M,N,K", [(8, 384, 25600), (3, 5120, 25600), (4, 256, 16640)])
def test_shapes_two_launches(M, N, K):
    """M * K above the one-launch limit: quantized into the workspace, then the GEMV."""
    assert M * K > 65536
    _check(M, N, K, seed=M * 17 + N, oracle=N <= 384)


def test_more_chunks_than_a_cta_holds():
    """M = 1, K = 65536 (256 chunks) over 40 tiles: a CTA would need more than 24 chunks, so two launches."""
    _check(1, 5120, 65536, seed=3)


def test_zero_and_tiny_activations():
    M, N, K = 4, 700, 1024
    y = _check(M, N, K, seed=5, x=torch.zeros(M, K, dtype=torch.bfloat16))
    assert not y.any()
    x = synth.activations(M, K, 6)
    x[1] = 0
    x[2] *= 1e-30          # block scales underflow relative to the tensor maximum
    _check(M, N, K, seed=6, x=x, oracle=True)


@pytest.mark.parametrize("name,K,N", synth.QWEN3_32B)
def test_full_size_bits_at_every_m(name, K, N):
    """Full-size Qwen3-32B projections: the one call gives the two calls' bits at M = 1..8."""
    w = synth.weights(N, K, seed=779)
    P = api.nvfp4_pack_weights(api.nvfp4_quantize_act(w.cuda()))
    ws = torch.zeros(api.nvfp4_quantize_gemv_workspace_bytes(8, N, K), dtype=torch.uint8, device="cuda")
    for M in range(1, 9):
        x = synth.activations(M, K, seed=920 + M).cuda()
        y = to_np(api.nvfp4_quantize_gemv_packed(x, P, workspace=ws))
        y2, _ = _two_calls(x, P, M, N, K)
        assert np.array_equal(y.view(np.uint32), y2.view(np.uint32)), (name, M)


def test_back_to_back_on_one_workspace_and_graph():
    """Calls of different shapes queued on one workspace, eagerly and replayed
    from a CUDA graph, give the bits of isolated calls."""
    shapes = [(8, 10240, 5120), (1, 1000, 768), (4, 5120, 8192), (8, 51200, 512), (2, 384, 25600), (1, 129, 256)]
    ops = []
    for i, (M, N, K) in enumerate(shapes):
        x = synth.activations(M, K, 80 + i).cuda()
        P = api.nvfp4_pack_weights(api.nvfp4_quantize_act(synth.weights(N, K, 90 + i).cuda()))
        ops.append((x, P, _two_calls(x, P, M, N, K)[0]))
    need = max(api.nvfp4_quantize_gemv_workspace_bytes(M, N, K) for M, N, K in shapes)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    ys = [torch.empty(x.shape[0], P.N, dtype=torch.float32, device="cuda") for x, P, _ in ops]
    for _ in range(2):
        for (x, P, _), y in zip(ops, ys):
            api.nvfp4_quantize_gemv_packed(x, P, y=y, workspace=ws)
        for (_, _, ref), y in zip(ops, ys):
            assert np.array_equal(to_np(y).view(np.uint32), ref.view(np.uint32))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for (x, P, _), y in zip(ops, ys):
                api.nvfp4_quantize_gemv_packed(x, P, y=y, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    for y in ys:
        y.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for (_, _, ref), y in zip(ops, ys):
        assert np.array_equal(to_np(y).view(np.uint32), ref.view(np.uint32))
    assert api.device_status() == 0


_CHILD = r"""
import numpy as np, torch
from nvfp4_w4a4_decode_gemv_gb300 import api, synth
for i, (M, N, K) in enumerate([(8, 51200, 5120), (8, 10240, 5120), (6, 5120, 8192), (3, 3000, 2816)]):
    x = synth.activations(M, K, 300 + i).cuda()
    P = api.nvfp4_pack_weights(api.nvfp4_quantize_act(synth.weights(N, K, 400 + i).cuda()))
    y = api.nvfp4_quantize_gemv_packed(x, P)
    X = api.nvfp4_quantize_act(x)
    y2 = api.nvfp4_gemv_smallm_packed(X, P)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), y2.view(torch.int32)), (M, N, K)
assert api.device_status() == 0
print("ok")
"""


def test_one_launch_beyond_the_default_block_limit():
    """With the limits raised (a fresh process reads the knobs), CTAs that
    quantize more blocks than their registers hold (the reload loop) and the
    Qwen3-32B gate_up at M = 8 run in one launch and still give the two calls' bits."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, NVFP4_QGEMV_MAX_BLOCKS="100000", NVFP4_QGEMV_MAX_M="8")
    r = subprocess.run([sys.executable, "-c", _CHILD], cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr


def test_launch_query():
    """nvfp4_quantize_gemv_launches: one launch for the Qwen3-32B shapes at M <= 3
    (except down at M = 3, M * K above the limit), two above, 0 for bad shapes."""
    for name, K, N in synth.QWEN3_32B:
        for M in range(1, 9):
            want = 1 if M <= 3 and M * K <= 65536 else 2
            assert api.nvfp4_quantize_gemv_launches(M, N, K) == want, (name, M)
    assert api.nvfp4_quantize_gemv_launches(1, 5120, 65536) == 2        # 34 chunks a CTA
    assert api.nvfp4_quantize_gemv_launches(9, 5120, 5120) == 0
