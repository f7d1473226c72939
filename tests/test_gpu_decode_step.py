"""The synthetic Qwen3-32B decode step (2 layers, full-size shapes) vs the oracle,
stage by stage: every stage is recomputed by the oracle from the GPU's own
input to that stage, so each kernel of the chain is checked at its own bar.

* RMS norm: BF16 equal to the exact value's rounding, except within 8 FP32
  ulps of a rounding boundary (either neighbour then).
* Quantizers on BF16 / FP32 rows: codes, scales and global scale bit-exact.
* SiLU*mul quantizer: exact on blocks whose 16 values are decisive (see
  tests/test_gpu_quantize.py).
* NVFP4 GEMVs: 48 sampled output rows per projection within
  1e-3 * sum |x w| + 1e-6; the lm_head (BF16) within 1e-4 * sum |x w| + 1e-6.
* Sampler: H within 1e-4 relative, T exact outside the guard band, token in
  the oracle's set of tokens whose CDF lies within 4e-6 Z of u Z.

Eager runs and graph replays of the same step give the same bits in every
intermediate buffer.
"""
import numpy as np
import pytest
import torch

from oracle import decode as D
from oracle import nvfp4 as Q
from oracle import reset as R
from nvfp4_w4a4_decode_gemv_gb300 import api, synth
from nvfp4_w4a4_decode_gemv_gb300.decode_step import DecodeStep
from tests.gpu_util import assert_within, bits, to_np

pytestmark = pytest.mark.gpu

EPS = 1e-6
ROWS = 48


def _check_norm(h_in, r_gpu):
    a = D.rms_norm(h_in, EPS)
    mid = D.to_bf16_bits(a)
    lo = D.to_bf16_bits(a * (1 - 8 * 2.0 ** -24))
    hi = D.to_bf16_bits(a * (1 + 8 * 2.0 ** -24))
    dec = (lo == hi) & (lo == mid)
    assert dec.mean() > 0.99
    got = bits(r_gpu)
    assert np.array_equal(got[dec], mid[dec])
    assert np.all((got[~dec] == lo[~dec]) | (got[~dec] == hi[~dec]))


def _check_quant(x_bf16_bits, traced):
    rc, rs, rg = Q.quantize_bf16(x_bf16_bits)
    codes, scales, g = (to_np(t) for t in traced)
    assert np.array_equal(codes, rc) and np.array_equal(scales, rs) and g[0] == rg


def _check_gemv(x_bf16_bits, w_rowmajor, y_gpu, rng):
    """y_gpu [M, N] vs the oracle on sampled rows, from the oracle's own codes of
    the GPU's BF16 input (those are bit-identical to the GPU's, checked by the
    quantizer stages)."""
    xq, xs, xg = Q.quantize_bf16(x_bf16_bits)
    N = y_gpu.shape[1]
    rows = np.unique(np.concatenate([rng.choice(N, ROWS, replace=False), [0, N - 1]]))
    wq = to_np(w_rowmajor.codes)[rows]
    ws = to_np(w_rowmajor.scales)[rows]
    wg = to_np(w_rowmajor.global_scale)[0]
    y_ref, bound = Q.gemv(xq, xs, xg, wq, ws, wg)
    assert_within(to_np(y_gpu)[:, rows], y_ref, bound)


@pytest.fixture(scope="module")
def step():
    st = DecodeStep(M=4, layers=2, keep_rowmajor=True, seed=1)
    st.h_in.copy_(synth.activations(4, st.hidden, seed=11).float().cuda())
    st.step_start.fill_(1)
    st.u.copy_(torch.tensor([0.1, 0.5, 0.9, 0.999], dtype=torch.float32))
    return st


def _check_layer(step, tr, wr, rng):
    """Every stage of one traced layer against the oracle, each from the GPU's
    own input to that stage."""
    _check_norm(to_np(tr["h_in"]), tr["r"])
    r_bits = bits(tr["r"])
    _check_quant(r_bits, tr["xq"])
    _check_gemv(r_bits, wr["qkv"], tr["y_qkv"], rng)
    q_bits = Q.f32_to_bf16_bits(to_np(tr["y_qkv"])[:, :step.k_o])
    _check_quant(q_bits, tr["xq_o"])
    _check_gemv(q_bits, wr["o"], tr["y_o"], rng)
    _check_norm(to_np(tr["y_o"]), tr["r2"])
    _check_quant(bits(tr["r2"]), tr["xq_gu"])
    _check_gemv(bits(tr["r2"]), wr["gate_up"], tr["y_gu"], rng)
    # SiLU(gate) * up -> NVFP4: exact on decisive blocks
    gu = to_np(tr["y_gu"]).astype(np.float64)
    a = D.silu_mul(gu)
    mid = D.to_bf16_bits(a)
    dec = (D.to_bf16_bits(a * (1 - 8 * 2.0 ** -24)) == D.to_bf16_bits(a * (1 + 8 * 2.0 ** -24))) & \
          (D.to_bf16_bits(a * (1 + 8 * 2.0 ** -24)) == mid)
    rc, rs, rg = Q.quantize_bf16(mid)
    codes, scales, g = (to_np(t) for t in tr["xq_d"])
    amax_idx = np.unravel_index(np.argmax(np.abs(Q.bf16_bits_to_f32(mid))), mid.shape)
    if dec[amax_idx]:
        assert g[0] == rg
        blk = dec.reshape(step.M, -1, 16).all(axis=2)
        assert blk.mean() > 0.9
        assert np.array_equal(scales[blk], rs[blk])
        el = np.repeat(blk, 16, axis=1)
        assert np.array_equal(Q.unpack_codes(codes)[el], Q.unpack_codes(rc)[el])
    # down: the oracle multiplies the GPU's own codes (checked above)
    N = step.hidden
    rows = np.unique(np.concatenate([rng.choice(N, ROWS, replace=False), [0, N - 1]]))
    wd = wr["down"]
    y_ref, bound = Q.gemv(codes, scales, g[0], to_np(wd.codes)[rows], to_np(wd.scales)[rows],
                          to_np(wd.global_scale)[0])
    assert_within(to_np(tr["h_out"])[:, rows], y_ref, bound)


def _check_head(step, fin, tok, H, T, rng):
    """Final norm, lm_head (64 sampled vocabulary rows) and the sampler at the
    first position of a step, on the GPU's logits."""
    _check_norm(to_np(fin["h_final"]), fin["r_final"])
    V = step.vocab
    rows = rng.choice(V, 64, replace=False)
    ref, scale = D.bf16_gemv(bits(fin["r_final"]), bits(step.lm_head[rows]))
    logits = to_np(fin["logits"])
    assert_within(logits[:, rows], ref, scale, rel=1e-4)
    p = R.ResetParams(tau0=float(np.float32(0.6)), t_low=float(np.float32(0.3)), t_high=1.0, w=8)
    u = to_np(step.u)
    for r in range(step.M):
        ln = logits[r].astype(np.float64)
        Hr = R.token_entropy(ln)
        res = R.reset_update(R.RowState(w=8), Hr, True, p)
        assert abs(H[r] - Hr) <= 1e-4 * max(abs(Hr), 1e-6)
        if not R.temperature_is_ambiguous(res, p):
            assert T[r] == np.float32(res.T)
        lo, hi = R.acceptable_tokens(ln, float(T[r]), float(u[r]), 4e-6)
        assert lo <= tok[r] <= hi
    assert np.all(np.isfinite(logits))


def test_decode_step_stagewise(step):
    trace = []
    tok, H, T = step.run(trace=trace)
    tok, H, T = to_np(tok), to_np(H), to_np(T)
    rng = np.random.default_rng(7)
    for layer in range(step.layers):
        _check_layer(step, trace[layer], step.rowmajor[layer], rng)
    _check_head(step, trace[-1], tok, H, T, rng)
    assert api.device_status() == 0


def test_decode_step_full_depth_sampled():
    """The full 64-layer step (distinct random weights per layer, M = 1) at
    step 0: layers 0, 31 and 63 checked stage by stage, then the head."""
    st = DecodeStep(M=1, layers=64, keep_rowmajor=True, seed=3)
    st.h_in.copy_(synth.activations(1, st.hidden, seed=13).float().cuda())
    st.step_start.fill_(1)
    st.u.fill_(0.37)
    trace = []
    tok, H, T = st.run(trace=trace)
    tok, H, T = to_np(tok), to_np(H), to_np(T)
    rng = np.random.default_rng(8)
    for layer in (0, 31, 63):
        _check_layer(st, trace[layer], st.rowmajor[layer], rng)
    _check_head(st, trace[-1], tok, H, T, rng)
    assert api.device_status() == 0
    del st, trace
    torch.cuda.empty_cache()


def _buffers(st):
    torch.cuda.synchronize()
    return [t.clone() for t in (st.xq.codes, st.xq.global_scale, st.y_qkv, st.xq_o.codes, st.y_o, st.xq_gu.codes,
                                st.xq_gu.global_scale, st.y_gu, st.xq_d.codes, st.h, st.logits)]


def test_decode_step_graph_replay_matches_eager():
    """Eager runs and graph replays of a 3-layer step leave every intermediate
    buffer bit-identical.  The first eager run starts from uninitialised
    buffers, so a kernel that read its input before the preceding kernel had
    written it (a programmatic-launch hazard) would show here."""
    st = DecodeStep(M=8, layers=3, seed=2)
    st.h_in.copy_(synth.activations(8, st.hidden, seed=12).float().cuda())
    st.u.fill_(0.5)
    st.run()                                   # eager: sets kernel attributes, advances the sampler state
    first = _buffers(st)
    st.run()
    assert all(torch.equal(a, b) for a, b in zip(first, _buffers(st)))
    g = st.capture()
    for _ in range(2):
        g.replay()
        assert all(torch.equal(a, b) for a, b in zip(first, _buffers(st)))
    assert api.device_status() == 0


def test_decode_step_top_p_in_graph():
    """The decode step with the sliding-window threshold and top-p 0.95: the
    four top-p launches are captured with the rest of the step, a replay gives
    the eager tokens, and the tokens lie in the oracle's nucleus of the GPU's
    logits (lm_head only: no decoder layers)."""
    from nvfp4_w4a4_decode_gemv_gb300._lib import THRESHOLD_WINDOW, ResetParams
    rp = ResetParams(0.6, 0.3, 1.0, 8, THRESHOLD_WINDOW, 0.95)
    st = DecodeStep(M=8, layers=0, seed=4, reset=rp)
    st.h_in.copy_(synth.activations(8, st.hidden, seed=14).float().cuda())
    st.u.copy_(torch.from_numpy(synth.reset_uniforms(1, 8, seed=9)[0]).cuda())
    st.run()
    tok, H, T = (to_np(t).copy() for t in st.run())
    g = st.capture()
    g.replay()
    torch.cuda.synchronize()
    # every call sees the same logits, so the window holds copies of one H and
    # its mean is H (sums of up to 8 copies of an FP32 value are exact in FP64):
    # H < tau fails and T = T_high at every call, eager or replayed
    assert np.all(T == np.float32(1.0)) and np.all(to_np(st.sampler.T) == np.float32(1.0))
    assert np.array_equal(to_np(st.sampler.token), tok)
    logits = to_np(st.logits)
    u = to_np(st.u)
    for r in range(8):
        ln = logits[r].astype(np.float64)
        assert abs(H[r] - R.token_entropy(ln)) <= 1e-4 * abs(R.token_entropy(ln))
        ok = False
        for keep in R.nucleus_candidates(ln, 1.0, float(np.float32(0.95)), 1e-6):
            lo, hi = R.acceptable_tokens(ln, 1.0, float(u[r]), 4e-6, keep=keep)
            ok |= bool(lo <= tok[r] <= hi and keep[tok[r]])
        assert ok, r
    assert api.device_status() == 0
    del st, g
    torch.cuda.empty_cache()
