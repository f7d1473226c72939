"""GPU decode-step glue vs the oracle: the BF16 lm_head GEMV, the FP32 -> BF16
cast and the RMS normalization.

* BF16 GEMV: FP32 accumulation of at most K products, so
  |y - y_ref| <= 1e-4 * sum_k |x_k w_k| + 1e-6 (an FP32 sum of K terms in
  any order is within about K * 2^-24 of the exact sum, relative to the sum of
  magnitudes; each lane here sums K/256 terms, then a 32-lane tree).
* Cast: bit-exact against round-to-nearest-even.
* RMS norm: the kernel's FP32 sum of squares and its IEEE sqrt and division
  are within a few FP32 ulps of the exact value, so an element whose exact
  value lies within 8 FP32 ulps of a BF16 rounding boundary may take either
  BF16 neighbour; every other element must match exactly.
"""
import numpy as np
import pytest
import torch

from oracle import decode as D
from oracle import nvfp4 as Q
from nvfp4_w4a4_decode_gemv_gb300 import api, synth
from tests.gpu_util import assert_within, bits, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K", [(1, 1000, 512), (4, 4096, 5120), (8, 333, 6400), (3, 8, 8), (1, 77, 51200)])
def test_bf16_gemv(M, N, K):
    x = synth.activations(M, K, seed=M + N)
    w = synth.weights(N, K, seed=K)
    y = to_np(api.nvfp4_bf16_gemv(x.cuda(), w.cuda()))
    ref, scale = D.bf16_gemv(bits(x), bits(w))
    assert_within(y, ref, scale, rel=1e-4)


def test_bf16_gemv_lm_head_sampled_rows():
    """The decode step's lm_head shape (5120 -> 151936) at M = 8: the GPU computes
    all logits, the oracle checks 64 sampled vocabulary rows."""
    M, K, V = 8, 5120, synth.LM_HEAD_VOCAB
    x = synth.activations(M, K, seed=5, outliers=False)
    w = synth.weights(V, K, seed=6)
    y = to_np(api.nvfp4_bf16_gemv(x.cuda(), w.cuda()))
    rows = np.random.default_rng(1).choice(V, 64, replace=False)
    ref, scale = D.bf16_gemv(bits(x), bits(w[rows]))
    assert_within(y[:, rows], ref, scale, rel=1e-4)


def test_f32_to_bf16_bit_exact():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(4096, generator=g) * torch.logspace(-30, 30, 4096)
    y = api.nvfp4_f32_to_bf16(x.cuda())
    assert np.array_equal(bits(y), Q.f32_to_bf16_bits(x.numpy()))


def _decisive(a64, bf16_bits):
    lo = D.to_bf16_bits(a64 * (1 - 8 * 2.0 ** -24))
    hi = D.to_bf16_bits(a64 * (1 + 8 * 2.0 ** -24))
    return (lo == hi) & (lo == bf16_bits)


@pytest.mark.parametrize("rows,K,ld", [(1, 5120, 5120), (8, 5120, 5120), (4, 8192, 10240), (3, 25600, 25600), (2, 4, 4)])
def test_rms_norm(rows, K, ld):
    g = torch.Generator().manual_seed(rows * K)
    x = torch.randn((rows, ld), generator=g) * 3.0
    x[:, :: max(1, K // 50)] *= 20.0                                    # outlier columns
    out = api.nvfp4_rms_norm_bf16(x.cuda(), K=K, eps=1e-6)
    a = D.rms_norm(x[:, :K].numpy(), 1e-6)
    mid = D.to_bf16_bits(a)
    dec = _decisive(a, mid)
    assert dec.mean() > 0.99
    got = bits(out)
    assert np.array_equal(got[dec], mid[dec])
    # the rest are one of the two neighbours of the exact value
    nd = ~dec
    lo = D.to_bf16_bits(a * (1 - 8 * 2.0 ** -24))[nd]
    hi = D.to_bf16_bits(a * (1 + 8 * 2.0 ** -24))[nd]
    assert np.all((got[nd] == lo) | (got[nd] == hi))


def test_rms_norm_zero_row_and_eps():
    x = torch.zeros((2, 64))
    x[1] = 2.0
    out = Q.bf16_bits_to_f32(bits(api.nvfp4_rms_norm_bf16(x.cuda(), eps=0.25)))
    assert np.all(out[0] == 0)
    assert np.all(out[1] == Q.bf16_bits_to_f32(D.to_bf16_bits(np.full(64, 2 / np.sqrt(4.25)))))


def _rms_input(rows, K, ld):
    g = torch.Generator().manual_seed(rows * K + 7)
    x = torch.randn((rows, ld), generator=g) * 3.0
    x[:, :: max(1, K // 50)] *= 20.0                                    # outlier columns
    return x


@pytest.mark.parametrize("rows,K,ld", [(1, 5120, 5120), (4, 5120, 5120), (8, 5120, 5120), (3, 16384, 16400),
                                       (2, 16, 16), (5, 8192, 10240), (7, 4000, 4004)])
def test_rms_norm_quantize(rows, K, ld):
    """The fused launch: its BF16 rows pass the RMS-norm check, and its codes,
    scales and global scale are exactly the quantizer's recipe on those rows."""
    x = _rms_input(rows, K, ld)
    r = torch.empty((rows, K), dtype=torch.bfloat16, device="cuda")
    q = api.nvfp4_rms_norm_quantize(x.cuda(), K=K, eps=1e-6, r_out=r)
    a = D.rms_norm(x[:, :K].numpy(), 1e-6)
    mid = D.to_bf16_bits(a)
    dec = _decisive(a, mid)
    assert dec.mean() > 0.99
    got = bits(r)
    assert np.array_equal(got[dec], mid[dec])
    nd = ~dec
    lo = D.to_bf16_bits(a * (1 - 8 * 2.0 ** -24))[nd]
    hi = D.to_bf16_bits(a * (1 + 8 * 2.0 ** -24))[nd]
    assert np.all((got[nd] == lo) | (got[nd] == hi))
    rc, rs, rg = Q.quantize_bf16(got)
    assert np.array_equal(to_np(q.codes), rc)
    assert np.array_equal(to_np(q.scales), rs)
    assert to_np(q.global_scale)[0] == rg
    # without r_out: the same codes
    q2 = api.nvfp4_rms_norm_quantize(x.cuda(), K=K, eps=1e-6)
    assert torch.equal(q2.codes, q.codes) and torch.equal(q2.scales, q.scales)
    assert torch.equal(q2.global_scale, q.global_scale)
    assert api.device_status() == 0


def test_rms_norm_quantize_matches_two_launches_where_rows_agree():
    """Against nvfp4_rms_norm_bf16 + nvfp4_quantize_act: the BF16 rows agree
    except where the exact value sits on a rounding boundary, and where they
    agree everywhere the codes agree too."""
    x = _rms_input(8, 5120, 5120).cuda()
    r = torch.empty((8, 5120), dtype=torch.bfloat16, device="cuda")
    q = api.nvfp4_rms_norm_quantize(x, eps=1e-6, r_out=r)
    r2 = api.nvfp4_rms_norm_bf16(x, eps=1e-6)
    same = bits(r) == bits(r2)
    assert same.mean() > 0.999
    if same.all():
        q2 = api.nvfp4_quantize_act(r2)
        assert torch.equal(q.codes, q2.codes) and torch.equal(q.scales, q2.scales)
        assert torch.equal(q.global_scale, q2.global_scale)


def test_rms_norm_quantize_zero_rows():
    x = torch.empty((0, 64), device="cuda")
    q = api.nvfp4_rms_norm_quantize(x)
    assert to_np(q.global_scale)[0] == 0.0


@pytest.mark.parametrize("M,N,K", [(1, 1000, 512), (4, 4096, 5120), (8, 333, 6400), (3, 8, 64), (8, 129, 25600),
                                   (2, 70000, 128), (5, 1, 8192)])
def test_bf16_gemv_tc(M, N, K):
    """The tensor-core BF16 GEMV against the FP64 oracle (several tiles, a
    ragged last tile, K down to one chunk), bit-identical on repeat calls."""
    x = synth.activations(M, K, seed=M + N + 1)
    w = synth.weights(N, K, seed=K + 1)
    xd, wd = x.cuda(), w.cuda()
    ws = torch.zeros(api.nvfp4_bf16_gemv_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    y = api.nvfp4_bf16_gemv_tc(xd, wd, workspace=ws)
    ref, scale = D.bf16_gemv(bits(x), bits(w))
    assert_within(to_np(y), ref, scale, rel=1e-4)
    y2 = api.nvfp4_bf16_gemv_tc(xd, wd, workspace=ws)
    assert torch.equal(y, y2)
    assert api.device_status() == 0


@pytest.mark.parametrize("M", [1, 8])
def test_bf16_gemv_tc_lm_head_sampled_rows(M):
    """The decode step's lm_head (5120 -> 151936): all logits on the GPU, 64
    sampled vocabulary rows (and the last) checked by the oracle; the
    CUDA-core path agrees within the same bound."""
    K, V = 5120, synth.LM_HEAD_VOCAB
    x = synth.activations(M, K, seed=15, outliers=False)
    w = synth.weights(V, K, seed=16)
    xd, wd = x.cuda(), w.cuda()
    y = to_np(api.nvfp4_bf16_gemv_tc(xd, wd))
    rows = np.concatenate([np.random.default_rng(2).choice(V, 64, replace=False), [V - 1]])
    ref, scale = D.bf16_gemv(bits(x), bits(w[rows]))
    assert_within(y[:, rows], ref, scale, rel=1e-4)
    ycc = to_np(api.nvfp4_bf16_gemv(xd, wd))
    full_scale = np.abs(to_np(xd.float())) @ np.abs(to_np(wd.float())).T
    assert np.all(np.abs(y - ycc) <= 2e-4 * full_scale + 2e-6)


def test_bf16_gemv_tc_shares_the_gemv_workspace():
    """BF16 and NVFP4 GEMV calls of different shapes back to back on one
    workspace: each still matches its own fresh-workspace result."""
    shapes = [(8, 5120, 10240), (1, 5120, 2048)]
    ws = torch.zeros(max(api.nvfp4_gemv_workspace_bytes(M, N, K) for M, K, N in shapes), dtype=torch.uint8,
                     device="cuda")
    outs = []
    for M, K, N in shapes:
        x = synth.activations(M, K, seed=N).cuda()
        w = synth.weights(N, K, seed=K).cuda()
        wq = api.nvfp4_quantize_act(w)
        xq = api.nvfp4_quantize_act(x)
        outs.append((api.nvfp4_bf16_gemv_tc(x, w, workspace=ws), api.nvfp4_gemv_smallm(xq, wq, workspace=ws),
                     api.nvfp4_bf16_gemv_tc(x, w), api.nvfp4_gemv_smallm(xq, wq)))
    for a, b, c, d in outs:
        assert torch.equal(a, c) and torch.equal(b, d)
    assert api.device_status() == 0
