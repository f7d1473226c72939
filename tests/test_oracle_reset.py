"""Pins for the oracle's ReSET entropy, state rule and sampler (no GPU).

Entropies are checked against closed forms; the state rule against a
hand-derived 11-position script (dyadic entropies, so every mean is exact);
the sampler against brute-force inverse CDFs on tiny vocabularies.
"""
import math

import numpy as np
import pytest

from oracle import reset as R


def test_entropy_uniform_is_log_v():
    for V in (2, 7, 151936):
        assert R.token_entropy(np.zeros(V)) == pytest.approx(math.log(V), rel=1e-12)
        assert R.token_entropy(np.full(V, 3.25)) == pytest.approx(math.log(V), rel=1e-12)


def test_entropy_two_level_closed_form():
    V, a = 1000, 2.5
    l = np.zeros(V)
    l[17] = a
    Z = math.exp(a) + (V - 1)
    want = math.log(Z) - a * math.exp(a) / Z
    # the oracle shifts by max = a: same value
    assert R.token_entropy(l) == pytest.approx(want, rel=1e-12)


def test_entropy_binary():
    a = 0.7
    p = 1 / (1 + math.exp(-a))
    want = -(p * math.log(p) + (1 - p) * math.log(1 - p))
    assert R.token_entropy(np.array([a, 0.0])) == pytest.approx(want, rel=1e-12)


def test_entropy_dominant_and_shift_invariant():
    l = np.zeros(5000)
    l[3] = 100.0
    eps = 4999 * math.exp(-100.0)                 # Z = 1 + eps after the shift by max
    want = math.log1p(eps) + 100.0 * eps / (1 + eps)
    assert R.token_entropy(l) == pytest.approx(want, rel=1e-9) and want < 2e-38
    rng = np.random.default_rng(0)
    x = rng.standard_normal(300) * 3
    assert R.token_entropy(x) == pytest.approx(R.token_entropy(x + 40.0), rel=1e-12)


def test_entropy_masked_logits_add_nothing():
    """-inf logits (masked tokens) have probability 0: the entropy is that of
    the remaining logits, e.g. the binary entropy for two finite ones."""
    a = 0.7
    p = 1 / (1 + math.exp(-a))
    want = -(p * math.log(p) + (1 - p) * math.log(1 - p))
    l = np.array([-np.inf, a, -np.inf, 0.0, -np.inf])
    assert R.token_entropy(l) == pytest.approx(want, rel=1e-12)
    rng = np.random.default_rng(1)
    x = rng.standard_normal(400) * 2
    m = x.copy()
    m[::3] = -np.inf
    assert R.token_entropy(m) == pytest.approx(R.token_entropy(x[np.isfinite(m)]), rel=1e-12)
    # masked tokens are never sampled
    assert all(np.isfinite(m[R.sample_inverse_cdf(m, 1.0, u)]) for u in (0.0, 0.3, 0.999))


@pytest.mark.parametrize("T,u,tok", [
    (1.0, 0.0, 0), (1.0, 0.05, 0), (1.0, 0.15, 1), (1.0, 0.35, 2), (1.0, 0.65, 3), (1.0, 0.999, 3),
    # T = 0.5 squares the probabilities: [1, 4, 9, 16] / 30 -> C = [1, 5, 14, 30] / 30
    (0.5, 0.02, 0), (0.5, 0.1, 1), (0.5, 0.4, 2), (0.5, 0.5, 3),
])
def test_sample_brute_force(T, u, tok):
    l = np.log(np.array([1.0, 2.0, 3.0, 4.0]))
    assert R.sample_inverse_cdf(l, T, u) == tok


def test_sample_low_temperature_and_ordering():
    l = np.array([0.0, 5.0, 4.9, -3.0])
    assert R.sample_inverse_cdf(l, 0.01, 0.5) == 1       # near-greedy
    # brute-force the CDF for a random tiny case
    rng = np.random.default_rng(1)
    for _ in range(200):
        V = int(rng.integers(1, 9))
        l = rng.standard_normal(V) * 2
        T = float(rng.choice([0.3, 1.0]))
        u = float(rng.uniform())
        p = np.exp((l - l.max()) / T)
        c = 0.0
        want = V - 1
        for i in range(V):
            c += p[i]
            if c > u * p.sum():
                want = i
                break
        lo, hi = R.acceptable_tokens(l, T, u, 1e-9)
        assert lo <= want <= hi
        assert R.sample_inverse_cdf(l, T, u) == want


# Hand-derived script, w = 3, tau0 = 0.6, T_low = 0.3, T_high = 1.0; steps start at t = 0 and 6.
SCRIPT_H = [1.0, 0.25, 0.5, 2.0, 0.5, 0.25, 1.5, 0.125, 1.0, 1.75, 0.875]
SCRIPT_START = [0, 0, 0, 0, 0, 0, 1, 0, 0, 0, 0]
#            H_step      H_bar        tau      T      j
SCRIPT_WANT = [
    (1.0,        1.0,        0.6,     1.0,  0),   # window [1]            confident
    (0.625,      0.625,      0.6,     0.3,  1),   # window [1,.25]        H < tau0
    (1.75 / 3,   1.75 / 3,   0.6,     0.3,  2),
    (0.9375,     0.9375,     0.6,     1.0,  3),   # j >= w: in-step mean
    (0.85,       0.85,       0.6,     0.3,  4),
    (0.75,       0.75,       0.6,     0.3,  5),
    (0.75,       6 / 7,      0.6,     1.0,  0),   # new step: window [.5,.25,1.5] crosses the start
    (0.625,      6.125 / 8,  0.6,     0.3,  1),
    (0.875,      7.125 / 9,  0.875,   1.0,  2),   # uncertain step: tau = H_step
    (1.09375,    0.8875,     1.09375, 1.0,  3),   # in-step mean of [1.5,.125,1,1.75]
    (1.05,       9.75 / 11,  1.05,    0.3,  4),   # H = .875 > tau0 but < tau -> T_low
]


def test_reset_rule_hand_script():
    p = R.ResetParams(tau0=0.6, t_low=0.3, t_high=1.0, w=3)
    st = R.RowState(w=3)
    for t, (H, s) in enumerate(zip(SCRIPT_H, SCRIPT_START)):
        res = R.reset_update(st, H, bool(s), p)
        hs, hb, tau, T, j = SCRIPT_WANT[t]
        assert res.j == j, t
        assert res.H_step == pytest.approx(hs, abs=1e-15), t
        assert res.H_bar == pytest.approx(hb, abs=1e-15), t
        assert res.tau == pytest.approx(tau, abs=1e-15), t
        assert res.T == T, t


def test_reset_every_position_a_new_step_uses_window():
    p = R.ResetParams(tau0=0.6, t_low=0.3, t_high=1.0, w=2)
    st = R.RowState(w=2)
    Hs = [0.5, 1.5, 0.25, 0.75]
    want = [0.5, 1.0, 0.875, 0.5]
    for H, wnt in zip(Hs, want):
        assert R.reset_update(st, H, True, p).H_step == wnt


def test_run_sequence_matches_rule_and_entropy():
    rng = np.random.default_rng(2)
    steps, M, V = 12, 3, 50
    logits = rng.standard_normal((steps, M, V)) * rng.choice([1, 3, 8], size=(steps, 1, 1))
    start = (rng.uniform(size=(steps, M)) < 0.3).astype(np.uint8)
    u = rng.uniform(size=(steps, M))
    p = R.ResetParams()
    res, toks = R.run_sequence(logits, start, u, p)
    for r in range(M):
        st = R.RowState(w=p.w)
        for t in range(steps):
            H = R.token_entropy(logits[t, r])
            one = R.reset_update(st, H, bool(start[t, r]), p)
            assert one.T == res[t][r].T and one.H == res[t][r].H
            assert toks[t, r] == R.sample_inverse_cdf(logits[t, r], one.T, u[t, r])


def test_ambiguity_detector():
    p = R.ResetParams()
    clear = R.StepResult(H=0.2, H_step=0.4, H_bar=0.9, tau=0.6, T=0.3, j=0)
    assert not R.temperature_is_ambiguous(clear, p)
    near_tau = R.StepResult(H=0.60001, H_step=0.4, H_bar=0.9, tau=0.6, T=1.0, j=0)
    assert R.temperature_is_ambiguous(near_tau, p)
    near_bar = R.StepResult(H=0.7, H_step=0.90001, H_bar=0.9, tau=0.90001, T=0.3, j=0)
    assert R.temperature_is_ambiguous(near_bar, p)


# ---- the two other threshold policies (reading note §3.1 Eq. (1), §6.3 Table 2) ----
# Same 11-position script.  Fixed: T_low exactly where H < tau0 = 0.6.
SCRIPT_T_FIXED = [1.0, 0.3, 0.3, 1.0, 0.3, 0.3, 1.0, 0.3, 1.0, 1.0, 1.0]
# Sliding window, w = 3: tau = mean of the last 3 entropies including H (the
# step boundary at t = 6 plays no part), worked by hand.
SCRIPT_TAU_WINDOW = [1.0, 0.625, 1.75 / 3, 2.75 / 3, 1.0, 2.75 / 3, 0.75, 0.625, 0.875, 2.875 / 3, 3.625 / 3]
SCRIPT_T_WINDOW = [1.0, 0.3, 0.3, 1.0, 0.3, 0.3, 1.0, 0.3, 1.0, 1.0, 0.3]


@pytest.mark.parametrize("policy", ["fixed", "window"])
def test_threshold_policies_hand_script(policy):
    p = R.ResetParams(tau0=0.6, t_low=0.3, t_high=1.0, w=3, threshold=policy)
    st = R.RowState(w=3)
    for t, (H, s) in enumerate(zip(SCRIPT_H, SCRIPT_START)):
        res = R.reset_update(st, H, bool(s), p)
        # the HSE estimate and the running mean are tracked whatever the policy
        hs, hb, _, _, j = SCRIPT_WANT[t]
        assert res.j == j and res.H_step == pytest.approx(hs, abs=1e-15) and res.H_bar == pytest.approx(hb, abs=1e-15)
        if policy == "fixed":
            assert res.tau == 0.6 and res.T == SCRIPT_T_FIXED[t], t
        else:
            assert res.tau == pytest.approx(SCRIPT_TAU_WINDOW[t], abs=1e-15), t
            assert res.T == SCRIPT_T_WINDOW[t], t


def test_unknown_policy_is_an_error():
    with pytest.raises(ValueError):
        R.reset_update(R.RowState(w=2), 0.5, False, R.ResetParams(threshold="ema"))


def test_policy_ambiguity_ignores_step_comparison_outside_reset():
    # H_step == H_bar is a guard-band case for ReSET only (tau0 = 0.6 gives
    # T_high at H = 0.7, tau = H_step = 0.9 gives T_low)
    res = R.StepResult(H=0.7, H_step=0.9, H_bar=0.9, tau=0.6, T=1.0, j=0)
    assert R.temperature_is_ambiguous(res, R.ResetParams(tau0=0.6, t_low=0.3))
    assert not R.temperature_is_ambiguous(res, R.ResetParams(tau0=0.6, t_low=0.3, threshold="fixed"))


# ---- top-p (reading note §6.1, §6.3 Table 5) ------------------------------------
@pytest.mark.parametrize("top_p,keep", [
    (0.49, [1]), (0.51, [1, 2]), (0.79, [1, 2]), (0.81, [0, 1, 2]), (1.0, [0, 1, 2]),
])
def test_nucleus_hand_worked(top_p, keep):
    # probabilities 0.2, 0.5, 0.3 in vocabulary order
    l = np.log(np.array([0.2, 0.5, 0.3]))
    assert np.flatnonzero(R.nucleus_mask(l, 1.0, top_p)).tolist() == keep


def test_nucleus_keeps_whole_tie_group():
    l = np.log(np.array([0.3, 0.4, 0.3]))
    assert R.nucleus_mask(l, 1.0, 0.5).tolist() == [True, True, True]     # 0.4 + one 0.3 reaches 0.5: both 0.3 stay
    assert R.nucleus_mask(l, 1.0, 0.39).tolist() == [False, True, False]
    assert R.nucleus_mask(np.zeros(10), 1.0, 0.01).all()                   # uniform: one group


def test_nucleus_temperature_applies_first():
    # p = [1, 2, 3, 4] / 10 at T = 1; at T = 0.5 they become [1, 4, 9, 16] / 30
    l = np.log(np.array([1.0, 2.0, 3.0, 4.0]))
    assert np.flatnonzero(R.nucleus_mask(l, 1.0, 0.5)).tolist() == [2, 3]   # 0.4 < 0.5 <= 0.7
    assert np.flatnonzero(R.nucleus_mask(l, 0.5, 0.5)).tolist() == [3]      # 16/30 >= 0.5
    assert np.flatnonzero(R.nucleus_mask(l, 0.5, 0.6)).tolist() == [2, 3]   # 16/30 < 0.6 <= 25/30


def _brute_nucleus(prob, top_p):
    """Smallest subset reaching top_p, by enumeration (distinct probabilities:
    the most massive subset of the smallest size that reaches top_p)."""
    import itertools
    V = len(prob)
    tot = prob.sum()
    for k in range(1, V + 1):
        best = max(itertools.combinations(range(V), k), key=lambda c: prob[list(c)].sum())
        if prob[list(best)].sum() >= top_p * tot:
            return sorted(best)
    return list(range(V))


def test_nucleus_brute_force_and_sample():
    rng = np.random.default_rng(7)
    n = 0
    for _ in range(300):
        V = int(rng.integers(1, 8))
        l = rng.standard_normal(V) * 2
        T = float(rng.choice([0.3, 1.0]))
        top_p = float(rng.uniform(0.05, 1.0))
        prob = np.exp((l - l.max()) / T)
        keep = _brute_nucleus(prob, top_p)
        if any(abs(prob[keep[:i]].sum() - top_p * prob.sum()) < 1e-9 for i in range(len(keep) + 1)):
            continue                                  # too close to a boundary for an exact comparison
        assert np.flatnonzero(R.nucleus_mask(l, T, top_p)).tolist() == keep
        # inverse CDF over the kept tokens only, renormalised
        u = float(rng.uniform())
        c, want = 0.0, keep[-1]
        for i in keep:
            c += prob[i]
            if c > u * prob[keep].sum():
                want = i
                break
        assert R.sample_inverse_cdf(l, T, u, top_p) == want
        n += 1
    assert n > 250


def test_nucleus_candidates_cover_boundary_groups():
    l = np.log(np.array([0.2, 0.5, 0.3]))
    # top_p * Z at exactly the kept mass 0.8: within rel of the group at 0.2
    c = R.nucleus_candidates(l, 1.0, 0.8 + 1e-9, 1e-6)
    masks = sorted(tuple(m.tolist()) for m in c)
    assert (True, True, True) in masks and (False, True, True) in masks
    assert len(R.nucleus_candidates(l, 1.0, 0.7, 1e-6)) == 1
    assert R.nucleus_candidates(l, 1.0, 1.0, 1e-6)[0].all()
