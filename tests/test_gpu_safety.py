"""Failure handling and out-of-bounds checks on the GPU, without any fault.

1. A GEMV CTA's bounded wait for another CTA's partial sum is made to run out
   through the library's test hook (partial sums are not published and the
   poll limit is short): the kernel returns, device error bit 2 is reported,
   the records it waited on are left zero, and the next call on the same
   workspace (zeroed again, as the header asks after that error) matches the
   oracle.
2. Output canaries, in place of a memory checker: every output is a view in
   the middle of a buffer whose 4 KB on each side hold a known byte pattern;
   after the call on ragged shapes (N = 1, 129, 1000; K = 16, 4112, 25616;
   V = 1, 2049, 4101) the guard bytes must be unchanged and the outputs must
   match the oracle.
"""
import numpy as np
import pytest
import torch

from oracle import decode as D
from oracle import nvfp4 as Q
from oracle import reset as R
from nvfp4_w4a4_decode_gemv_gb300 import api, synth
from nvfp4_w4a4_decode_gemv_gb300._lib import ResetParams, lib
from tests.gpu_util import Guarded, assert_within, bits, to_np

pytestmark = pytest.mark.gpu

def _guarded_nvfp4(rows, K):
    c, s, g = Guarded((rows, K // 2), torch.uint8), Guarded((rows, K // 16), torch.uint8), Guarded((1,), torch.float32)
    return (c, s, g), api.NVFP4Tensor(c.t, s.t, g.t)


# ---- 1. a bounded wait that runs out -------------------------------------------------------
@pytest.mark.parametrize("path", ["rowmajor", "packed", "one-call"])
def test_gemv_fixup_wait_runs_out_and_is_reported(path):
    M, N, K = 2, 1000, 768            # 24 units: one per CTA, every tile split three ways
    x, w = synth.activations(M, K, 31), synth.weights(N, K, 32)
    X, W = api.nvfp4_quantize_act(x.cuda()), api.nvfp4_quantize_act(w.cuda())
    Wp = api.nvfp4_pack_weights(W) if path != "rowmajor" else W
    xd = x.cuda()
    gemv = {"rowmajor": lambda ws: api.nvfp4_gemv_smallm(X, Wp, workspace=ws),
            "packed": lambda ws: api.nvfp4_gemv_smallm_packed(X, Wp, workspace=ws),
            # M = 2: the GEMV that quantizes its activation, one launch
            "one-call": lambda ws: api.nvfp4_quantize_gemv_packed(xd, Wp, workspace=ws)}[path]
    wsp = api.GemvWorkspace()
    ws = wsp.get_bytes(api.nvfp4_quantize_gemv_workspace_bytes(M, N, K))
    torch.cuda.synchronize()
    assert api.device_status() == 0
    L = lib()
    L.nvfp4_test_gemv_fault(1 << 10, 1)
    try:
        gemv(ws)
        torch.cuda.synchronize()      # the kernel returned: the wait gave up
    finally:
        L.nvfp4_test_gemv_fault(0, 0)
    assert int(torch.count_nonzero(ws)) == 0, "the timed-out reader left record words behind"
    assert api.device_status() == api.DEVERR_FLAG_TIMEOUT
    assert api.device_status() == 0
    y = to_np(gemv(ws))
    xq, xs, xg = Q.quantize_bf16(bits(x))
    wq, wsc, wg = Q.quantize_bf16(bits(w))
    y_ref, bound = Q.gemv(xq, xs, xg, wq, wsc, wg)
    assert_within(y, y_ref, bound)
    assert api.device_status() == 0


# ---- 2. output canaries ---------------------------------------------------------------------
@pytest.mark.parametrize("rows,K", [(1, 16), (3, 16), (5, 4112), (8, 25616)])
def test_quantizer_canaries(rows, K):
    x = synth.activations(rows, K, seed=rows * 7 + K)
    guards, out = _guarded_nvfp4(rows, K)
    api.nvfp4_quantize_act(x.cuda(), out=out)
    for gd, name in zip(guards, ("codes", "scales", "global")):
        gd.check(name)
    xq, xs, xg = Q.quantize_bf16(bits(x))
    assert np.array_equal(to_np(out.codes), xq) and np.array_equal(to_np(out.scales), xs)
    assert to_np(out.global_scale)[0] == xg


def test_quantizer_grid_path_canaries():
    """A weight-sized tensor (the multi-launch path) with a ragged K."""
    rows, K = 1000, 25616
    w = synth.weights(rows, K, seed=5)
    guards, out = _guarded_nvfp4(rows, K)
    api.nvfp4_quantize_act(w.cuda(), out=out)
    for gd, name in zip(guards, ("codes", "scales", "global")):
        gd.check(name)
    wf = Q.bf16_bits_to_f32(bits(w))
    g = Q.global_scale(wf)
    assert to_np(out.global_scale)[0] == g
    sample = np.array([0, 1, 517, rows - 1])
    wq, wsc, _ = Q.quantize_f32(wf[sample], g=g)
    assert np.array_equal(to_np(out.codes)[sample], wq) and np.array_equal(to_np(out.scales)[sample], wsc)


def test_glue_quantizer_canaries():
    """The decode step's fused quantizers on ragged widths.  SiLU uses the
    device expf, so its values are compared to the oracle only in bulk here
    (the quantizer tests check them element by element); the fused RMS norm +
    quantize is checked exactly against the oracle's quantization of its own
    BF16 output."""
    rows, inter, hidden = 3, 4112, 2064
    gu = torch.randn((rows, 2 * inter), generator=torch.Generator().manual_seed(3))
    guards, out = _guarded_nvfp4(rows, inter)
    api.nvfp4_silu_mul_quantize(gu.cuda(), out=out)
    for gd, name in zip(guards, ("codes", "scales", "global")):
        gd.check("silu_mul " + name)
    _, rs, _ = Q.quantize_bf16(D.to_bf16_bits(D.silu_mul(gu.numpy().astype(np.float64))))
    assert np.mean(to_np(out.scales) == rs) > 0.95
    h = torch.randn((rows, hidden), generator=torch.Generator().manual_seed(4))
    guards2, out2 = _guarded_nvfp4(rows, hidden)
    r = Guarded((rows, hidden), torch.bfloat16)
    api.nvfp4_rms_norm_quantize(h.cuda(), eps=1e-6, out=out2, r_out=r.t)
    for gd, name in zip(guards2 + (r,), ("codes", "scales", "global", "r_out")):
        gd.check("rms_norm_quantize " + name)
    rq, rsc, rg = Q.quantize_bf16(bits(r.t.cpu()))
    assert np.array_equal(to_np(out2.codes), rq) and np.array_equal(to_np(out2.scales), rsc)
    assert to_np(out2.global_scale)[0] == rg


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (3, 129, 256), (8, 1000, 768), (2, 129, 25856)])
@pytest.mark.parametrize("path", ["tc", "packed", "cc"])
def test_gemv_canaries(M, N, K, path):
    x, w = synth.activations(M, K, seed=N + K), synth.weights(N, K, seed=N + K + 1)
    X, W = api.nvfp4_quantize_act(x.cuda()), api.nvfp4_quantize_act(w.cuda())
    y = Guarded((M, N), torch.float32)
    if path == "packed":
        need = api.nvfp4_packed_weight_bytes(N, K)
        P = Guarded((need,), torch.uint8)
        Wp = api.nvfp4_pack_weights(W, out=P.t)
        P.check("packed weights")
        api.nvfp4_gemv_smallm_packed(X, Wp, y=y.t)
    elif path == "tc":
        api.nvfp4_gemv_smallm(X, W, y=y.t)
    else:
        api.nvfp4_gemv_smallm_cudacore(X, W, y=y.t)
    y.check("y")
    xq, xs, xg = Q.quantize_bf16(bits(x))
    wq, wsc, wg = Q.quantize_bf16(bits(w))
    y_ref, bound = Q.gemv(xq, xs, xg, wq, wsc, wg)
    assert_within(to_np(y.t), y_ref, bound)
    assert api.device_status() == 0


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (3, 129, 256), (2, 129, 25856), (8, 1000, 768)])
def test_quantize_gemv_canaries(M, N, K):
    """nvfp4_quantize_gemv_packed into guarded y and global-scale buffers (one
    launch for M <= 3 except where M * K is too large, two launches above)."""
    x, w = synth.activations(M, K, seed=N + K + 2), synth.weights(N, K, seed=N + K + 3)
    P = api.nvfp4_pack_weights(api.nvfp4_quantize_act(w.cuda()))
    y, g = Guarded((M, N), torch.float32), Guarded((1,), torch.float32)
    api.nvfp4_quantize_gemv_packed(x.cuda(), P, y=y.t, xg_out=g.t)
    y.check("y")
    g.check("global scale")
    xq, xs, xg = Q.quantize_bf16(bits(x))
    wq, wsc, wg = Q.quantize_bf16(bits(w))
    assert to_np(g.t)[0] == xg
    y_ref, bound = Q.gemv(xq, xs, xg, wq, wsc, wg)
    assert_within(to_np(y.t), y_ref, bound)
    assert api.device_status() == 0


@pytest.mark.parametrize("M,N,K", [(3, 129, 64), (8, 1000, 320), (1, 1, 128)])
def test_bf16_gemv_tc_canaries(M, N, K):
    g = torch.Generator().manual_seed(M + N + K)
    x = torch.randn((M, K), generator=g).to(torch.bfloat16)
    w = (torch.randn((N, K), generator=g) * 0.02).to(torch.bfloat16)
    y = Guarded((M, N), torch.float32)
    api.nvfp4_bf16_gemv_tc(x.cuda(), w.cuda(), y=y.t)
    y.check("y")
    y_ref, bound = D.bf16_gemv(bits(x), bits(w))
    assert_within(to_np(y.t), y_ref, bound, rel=1e-4)


@pytest.mark.parametrize("V", [1, 2049, 4101])
@pytest.mark.parametrize("top_p", [1.0, 0.9])
def test_sampler_canaries(V, top_p):
    M, w = 3, 8
    params = ResetParams(0.6, 0.3, 1.0, w, 0, top_p)
    state = torch.zeros(api.reset_state_bytes(M, w), dtype=torch.uint8, device="cuda")
    api.reset_state_init(state, M, w)
    ws = torch.zeros(api.reset_workspace_bytes(M, V), dtype=torch.uint8, device="cuda")
    tok, H, T = Guarded((M,), torch.int32), Guarded((M,), torch.float32), Guarded((M,), torch.float32)
    us = synth.reset_uniforms(3, M, seed=V)
    p = R.ResetParams(top_p=float(np.float32(top_p)))
    states = [R.RowState(w=w) for _ in range(M)]
    for t in range(3):
        logits = synth.reset_logits(t, M, V, 3.0)
        api.reset_sample(logits.cuda(), None, torch.from_numpy(us[t]).cuda(), state, params, tok.t, H.t, T.t, ws)
        for gd, name in ((tok, "token"), (H, "H"), (T, "T")):
            gd.check(name)
        ln = logits.numpy().astype(np.float64)
        for r in range(M):
            res = R.reset_update(states[r], R.token_entropy(ln[r]), t == 0, p)
            Tr = float(to_np(T.t)[r])
            if not R.temperature_is_ambiguous(res, p):
                assert Tr == np.float32(res.T)
            k = int(to_np(tok.t)[r])
            ok = False
            for keep in R.nucleus_candidates(ln[r], Tr, p.top_p, 1e-6):
                lo, hi = R.acceptable_tokens(ln[r], Tr, float(us[t, r]), 4e-6, keep=keep)
                ok = ok or (lo <= k <= hi and bool(keep[k]))
            assert ok, (V, t, r, k)
    assert api.device_status() == 0
