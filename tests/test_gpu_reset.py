"""GPU ReSET sampler vs the oracle over whole sequences.

Per row and position: H within 1e-4 relative; T equal unless the oracle's
comparison is inside its 1e-4 guard band (then either T is accepted); the
token equal to the oracle's inverse-CDF sample at the GPU's T, up to the
tokens whose cumulative sum lies within 4e-6 * Z of u * Z (the GPU sums exp
values of FP32 accuracy -- 2 ulp per exp, FP32 chunk sums of <= 2048 terms --
so its partial sums carry a relative error below that bound).  The same for
the fixed and sliding-window threshold policies and for top-p, where the
token must also lie in the oracle's nucleus (or, when the nucleus boundary is
within 1e-6 * Z, in the nucleus with the boundary group on the other side).

The band is a tolerance on the exact rule, not the rule: every run also counts
the positions whose token differs from the oracle's exact inverse-CDF pick at
the same T and u, and asserts that there is at most one such position per run
(u * Z falls within the GPU's ~1e-7 * Z error of a CDF step with probability
~1e-7 per position, so the expected count over the 2048 x 8 run is ~0.003).
"""
import numpy as np
import pytest
import torch

from oracle import reset as R
from nvfp4_w4a4_decode_gemv_gb300 import api, synth
from nvfp4_w4a4_decode_gemv_gb300._lib import ResetParams

pytestmark = pytest.mark.gpu

TOKEN_REL = 4e-6
# top-p: the kernels' integer masses carry the FP32 exp's error (a few ulp) and
# one rounding to 2^-(62 - ceil(log2 V)) of the maximum's mass each, so a
# boundary logit group within 1e-6 * Z of top_p * Z may fall either way.
NUCLEUS_REL = 1e-6


def _f32(v):
    return float(np.float32(v))


def _token_ok(ln, T, u, tok, top_p):
    """The token is the oracle's inverse-CDF sample at T up to TOKEN_REL * Z,
    over one of the nuclei the oracle's guard band allows (all tokens when
    top_p = 1), and is a member of that nucleus."""
    for keep in R.nucleus_candidates(ln, T, top_p, NUCLEUS_REL):
        lo, hi = R.acceptable_tokens(ln, T, u, TOKEN_REL, keep=keep)
        if lo <= tok <= hi and keep[tok]:
            return True
    return False


def _run(M, V, steps, sigmas, starts, us, tau0=0.6, t_low=0.3, t_high=1.0, w=8, seed0=4, pass_starts=True,
         threshold="reset", top_p=1.0):
    p_gpu = dict(tau0=tau0, t_low=t_low, t_high=t_high, w=w, threshold=threshold, top_p=top_p)
    sampler = api.ResetSampler(M, V, **p_gpu)
    p = R.ResetParams(tau0=_f32(tau0), t_low=_f32(t_low), t_high=_f32(t_high), w=w, threshold=threshold,
                      top_p=_f32(top_p))
    states = [R.RowState(w=w) for _ in range(M)]
    n_amb = 0
    n_inexact = 0                    # tokens accepted only through the TOKEN_REL / NUCLEUS_REL band
    for t in range(steps):
        logits = synth.reset_logits(t, M, V, float(sigmas[t]), base_seed=seed0)
        st = torch.from_numpy(starts[t]).cuda() if pass_starts else None
        u = torch.from_numpy(us[t]).cuda()
        tok, H, T = sampler(logits.cuda(), st, u)
        torch.cuda.synchronize()
        tok, H, T = tok.cpu().numpy(), H.cpu().numpy(), T.cpu().numpy()
        ln = logits.numpy().astype(np.float64)
        for r in range(M):
            Hr = R.token_entropy(ln[r])
            res = R.reset_update(states[r], Hr, bool(starts[t, r]) and pass_starts, p)
            assert abs(H[r] - Hr) <= 1e-4 * max(abs(Hr), 1e-6), (t, r, H[r], Hr)
            if R.temperature_is_ambiguous(res, p):
                n_amb += 1
                assert T[r] in (np.float32(t_low), np.float32(t_high))
            else:
                assert T[r] == np.float32(res.T), (t, r, T[r], res)
            assert _token_ok(ln[r], float(T[r]), float(us[t, r]), int(tok[r]), p.top_p), (t, r, tok[r])
            if int(tok[r]) != R.sample_inverse_cdf(ln[r], float(T[r]), float(us[t, r]), p.top_p):
                n_inexact += 1
    assert api.device_status() == 0
    assert n_inexact <= 1, f"{n_inexact} of {steps * M} tokens differ from the exact inverse-CDF pick"
    return n_amb


def test_small_vocab_sequence():
    M, V, steps = 8, 5000, 40
    _run(M, V, steps, synth.reset_sigmas(steps), synth.reset_boundaries(steps, M, p=0.15),
         synth.reset_uniforms(steps, M))


def test_full_size_sequence_prefix():
    """M = 8 rows x V = 151936 logits (the sampler workload), first 24 positions."""
    M, V, steps = 8, synth.LM_HEAD_VOCAB, 24
    _run(M, V, steps, synth.reset_sigmas(steps), synth.reset_boundaries(steps, M, p=1 / 4),
         synth.reset_uniforms(steps, M))


def test_long_sequence_2048_steps():
    """The sampler workload's length: M = 8 rows over 2048 positions, step
    boundaries with gaps ~ Geometric(1/30) (long steps exercise the in-step mean
    after the first w positions), sigma per position from {1, 3, 8}; V = 4096
    keeps the oracle fast -- the state rules do not depend on V, and the full
    vocabulary is covered by test_full_size_sequence_prefix."""
    M, V, steps = 8, 4096, 2048
    _run(M, V, steps, synth.reset_sigmas(steps), synth.reset_boundaries(steps, M), synth.reset_uniforms(steps, M))


@pytest.mark.parametrize("V", [1, 2, 2047, 2048, 2049, 4096 + 5])
def test_ragged_and_tiny_vocab(V):
    M, steps = 3, 6
    _run(M, V, steps, synth.reset_sigmas(steps, seed=V), synth.reset_boundaries(steps, M, p=0.3, seed=V),
         synth.reset_uniforms(steps, M, seed=V))


def test_no_step_flags_and_other_params():
    M, V, steps = 4, 3000, 20
    _run(M, V, steps, synth.reset_sigmas(steps, seed=1), synth.reset_boundaries(steps, M, p=0.2, seed=1),
         synth.reset_uniforms(steps, M, seed=1), tau0=0.5, t_low=0.1, t_high=1.0, w=3, pass_starts=False)


def test_u_zero_gives_first_token_with_mass():
    M, V = 2, 100
    sampler = api.ResetSampler(M, V)
    logits = torch.zeros((M, V))
    logits[0, :10] = -200.0          # exp underflows to 0 at T = 0.3 and T = 1 in FP32
    tok, _, _ = sampler(logits.cuda(), None, torch.zeros(M).cuda())
    torch.cuda.synchronize()
    assert tok.tolist() == [10, 0]


def test_repeatable_and_state_restart():
    M, V, steps = 4, 7000, 8
    sig, st, us = synth.reset_sigmas(steps), synth.reset_boundaries(steps, M, p=0.3), synth.reset_uniforms(steps, M)
    outs = []
    for _ in range(2):
        sampler = api.ResetSampler(M, V)
        toks = []
        for t in range(steps):
            tok, H, T = sampler(synth.reset_logits(t, M, V, float(sig[t])).cuda(), torch.from_numpy(st[t]).cuda(),
                                torch.from_numpy(us[t]).cuda())
            toks.append((tok.cpu().numpy().copy(), H.cpu().numpy().copy(), T.cpu().numpy().copy()))
        outs.append(toks)
    for a, b in zip(*outs):
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


def test_window_mismatch_is_reported_without_fault():
    """A call whose window differs from the state's records a device error; the
    context stays usable."""
    M, V = 2, 512
    sampler = api.ResetSampler(M, V, w=8)
    sampler.params = ResetParams(0.6, 0.3, 1.0, 4)
    sampler(torch.zeros((M, V)).cuda(), None, torch.zeros(M).cuda())
    torch.cuda.synchronize()
    assert api.device_status() == 2
    assert api.device_status() == 0


@pytest.mark.parametrize("threshold", ["fixed", "window"])
def test_threshold_policies_sequence(threshold):
    M, V, steps = 8, 5000, 40
    _run(M, V, steps, synth.reset_sigmas(steps, seed=2), synth.reset_boundaries(steps, M, p=0.15, seed=2),
         synth.reset_uniforms(steps, M, seed=2), w=3, threshold=threshold)


def test_top_p_full_size_prefix():
    """Top-p 0.95 (the pages' evaluation setting) on M = 8 rows x V = 151936
    logits, sigma from {1, 3, 8}: nuclei from one token to most of the
    vocabulary."""
    M, V, steps = 8, synth.LM_HEAD_VOCAB, 10
    _run(M, V, steps, synth.reset_sigmas(steps, seed=3), synth.reset_boundaries(steps, M, p=1 / 4, seed=3),
         synth.reset_uniforms(steps, M, seed=3), top_p=0.95)


@pytest.mark.parametrize("top_p", [1.0, 0.95])
def test_rows_longer_than_one_cluster(top_p):
    """V = 300001 > 8 x 1024 x 32: the multi-launch path (chunk partials, a
    last-CTA merge and, with top-p, the four nucleus launches)."""
    M, V, steps = 2, 300001, 4
    _run(M, V, steps, synth.reset_sigmas(steps, seed=15), synth.reset_boundaries(steps, M, p=0.3, seed=15),
         synth.reset_uniforms(steps, M, seed=15), top_p=top_p)


@pytest.mark.parametrize("top_p,threshold", [(0.5, "reset"), (0.9, "window"), (0.05, "fixed")])
@pytest.mark.parametrize("V", [1, 3, 2047, 2049, 6001])
def test_top_p_ragged_vocab(V, top_p, threshold):
    M, steps = 3, 6
    _run(M, V, steps, synth.reset_sigmas(steps, seed=V), synth.reset_boundaries(steps, M, p=0.3, seed=V),
         synth.reset_uniforms(steps, M, seed=V), top_p=top_p, threshold=threshold)


def _tie_logits(M, V, seed):
    """Integer logits in [-3, 1] (large tie groups), one -0.0 per row."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randint(-3, 2, (M, V), generator=g).float()
    x[:, 7] = -0.0
    return x


@pytest.mark.parametrize("top_p", [0.3, 0.7, 0.95])
def test_top_p_keeps_whole_tie_groups(top_p):
    M, V = 4, 9000
    sampler = api.ResetSampler(M, V, top_p=top_p)
    p = R.ResetParams(top_p=_f32(top_p))
    us = synth.reset_uniforms(8, M, seed=11)
    for t in range(8):
        logits = _tie_logits(M, V, seed=100 + t)
        tok, H, T = sampler(logits.cuda(), None, torch.from_numpy(us[t]).cuda())
        torch.cuda.synchronize()
        ln = logits.numpy().astype(np.float64)
        for r in range(M):
            assert _token_ok(ln[r], float(T.cpu()[r]), float(us[t, r]), int(tok.cpu()[r]), p.top_p)
    assert api.device_status() == 0


@pytest.mark.parametrize("top_p", [0.5, 0.95])
def test_top_p_tie_groups_full_vocab(top_p):
    """V = 151936 (eight CTAs a row, 512 gathered keys each): tie groups of
    ~30k logits fill one log-mass bin, more than the gather holds, so the
    boundary comes from the three-level radix search."""
    M, V = 2, synth.LM_HEAD_VOCAB
    sampler = api.ResetSampler(M, V, top_p=top_p)
    p = R.ResetParams(top_p=_f32(top_p))
    us = synth.reset_uniforms(3, M, seed=12)
    for t in range(3):
        logits = _tie_logits(M, V, seed=200 + t)
        tok, H, T = sampler(logits.cuda(), None, torch.from_numpy(us[t]).cuda())
        torch.cuda.synchronize()
        ln = logits.numpy().astype(np.float64)
        for r in range(M):
            assert _token_ok(ln[r], float(T.cpu()[r]), float(us[t, r]), int(tok.cpu()[r]), p.top_p)
    assert api.device_status() == 0


def test_top_p_bf16_valued_logits_full_vocab():
    """Logits rounded to BF16 (a model's output): ties of a few hundred per
    value, which the gather holds, across M = 8 rows of V = 151936."""
    M, V, steps = 8, synth.LM_HEAD_VOCAB, 3
    sampler = api.ResetSampler(M, V, top_p=0.95)
    p = R.ResetParams(top_p=_f32(0.95))
    us = synth.reset_uniforms(steps, M, seed=13)
    for t in range(steps):
        logits = synth.reset_logits(t, M, V, 2.0).to(torch.bfloat16).float()
        tok, H, T = sampler(logits.cuda(), None, torch.from_numpy(us[t]).cuda())
        torch.cuda.synchronize()
        ln = logits.numpy().astype(np.float64)
        for r in range(M):
            assert _token_ok(ln[r], float(T.cpu()[r]), float(us[t, r]), int(tok.cpu()[r]), p.top_p)
    assert api.device_status() == 0


@pytest.mark.parametrize("top_p", [1.0, 0.95])
def test_masked_logits_full_vocab(top_p):
    """-inf logits (masked tokens) add nothing to H or Z and are never
    sampled, including a CTA whose whole range is masked (rows 0 and 2: the
    last and the first 20480 logits of V = 151936)."""
    M, V, steps = 4, synth.LM_HEAD_VOCAB, 3
    sampler = api.ResetSampler(M, V, top_p=top_p)
    p = R.ResetParams(top_p=_f32(top_p))
    states = [R.RowState(w=8) for _ in range(M)]
    us = synth.reset_uniforms(steps, M, seed=14)
    for t in range(steps):
        logits = synth.reset_logits(t, M, V, 3.0)
        logits[0, 143360:] = -np.inf
        logits[1, ::5] = -np.inf
        logits[2, :20480] = -np.inf
        g = torch.Generator().manual_seed(t)
        logits[3][torch.rand(V, generator=g) < 0.5] = -np.inf
        tok, H, T = sampler(logits.cuda(), None, torch.from_numpy(us[t]).cuda())
        torch.cuda.synchronize()
        tok, H, T = tok.cpu().numpy(), H.cpu().numpy(), T.cpu().numpy()
        ln = logits.numpy().astype(np.float64)
        for r in range(M):
            Hr = R.token_entropy(ln[r])
            res = R.reset_update(states[r], Hr, t == 0, p)
            assert abs(H[r] - Hr) <= 1e-4 * max(abs(Hr), 1e-6), (t, r, H[r], Hr)
            if not R.temperature_is_ambiguous(res, p):
                assert T[r] == np.float32(res.T), (t, r, T[r], res)
            assert np.isfinite(ln[r, int(tok[r])]), (t, r, tok[r])
            assert _token_ok(ln[r], float(T[r]), float(us[t, r]), int(tok[r]), p.top_p), (t, r, tok[r])
    assert api.device_status() == 0


def test_top_p_single_token_nucleus_and_u_extremes():
    """One dominant logit: at top_p <= its probability only it is kept, for
    every u, including u = 0 and the largest float below 1."""
    M, V = 3, 4096
    logits = torch.zeros((M, V))
    logits[:, 1234] = 12.0
    for u0 in (0.0, float(np.nextafter(np.float32(1.0), np.float32(0.0)))):
        sampler = api.ResetSampler(M, V, top_p=0.5)
        tok, _, _ = sampler(logits.cuda(), None, torch.full((M,), u0).cuda())
        torch.cuda.synchronize()
        assert tok.tolist() == [1234] * M


def test_top_p_repeatable_and_noalloc_identical():
    """The top-p path is deterministic (integer masses), and the allocation-free
    entry point gives the same tokens."""
    M, V, steps = 8, 20000, 6
    sig, us = synth.reset_sigmas(steps, seed=5), synth.reset_uniforms(steps, M, seed=5)
    runs = []
    for noalloc in (False, False, True):
        sampler = api.ResetSampler(M, V, top_p=0.95, threshold="window")
        toks = []
        for t in range(steps):
            logits = synth.reset_logits(t, M, V, float(sig[t])).cuda()
            u = torch.from_numpy(us[t]).cuda()
            if noalloc:
                api.reset_sample_noalloc(logits, None, u, sampler.state, sampler.params, sampler.token, sampler.H,
                                         sampler.T)
            else:
                sampler(logits, None, u)
            toks.append(sampler.token.cpu().numpy().copy())
        runs.append(np.stack(toks))
    assert np.array_equal(runs[0], runs[1]) and np.array_equal(runs[0], runs[2])
    assert api.device_status() == 0
