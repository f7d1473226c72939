"""ReSET step-aware temperature sampling, plain and slow (FP64).

Sources (the ReSET pages):
  * token entropy H_t of the next-token distribution (project page, "Step-aware
    temperature scaling"; reading note §3.1);
  * a reasoning step is a span cut at a double newline and its entropy is the
    mean token entropy inside it (reading note §3.2);
  * SAT, the step-aware threshold: tau_t = tau0 when the step is confident
    (step estimate <= running global mean H_bar), else tau_t = the step
    estimate itself (reading note §4.1; project page formula);
  * HSE, the online step-entropy estimate: for the first w positions of a step
    the mean of the last w token entropies (crossing the step boundary), after
    that the running in-step mean (reading note §4.2);
  * T_t = T_low if H_t < tau_t else T_high (project page formula; reading note
    Eq. (1) in §3.1 and §4.3), then sample from softmax(logits / T_t);
  * the two threshold policies ReSET is compared against (reading note §3.1
    Eq. (1) and §6.3, Table 2): a fixed threshold tau_t = tau0, and a
    sliding-window threshold;
  * nucleus (top-p) truncation, which the pages' evaluation applies on top of
    the temperature (reading note §6.1 "top-p=0.95", §6.3 Table 5).

Readings where the pages leave a step open (each pinned by a test):
  * entropy is in nats, at temperature 1, of the raw logits;
  * step_start[r] = 1 at a call means this position is the FIRST position of a
    new step (the previous token was the double newline); position 0 of a
    sequence always starts a step;
  * both the window mean and the in-step mean include H_t itself; the window is
    truncated at the start of the sequence; "the first w positions" means the
    0-based in-step position j < w;
  * H_bar_t is the mean of H_0..H_t (including t);
  * the sample is inverse-CDF: token = min{ i : C_i > u * Z } with
    C_i = sum_{k<=i} exp(s_k / T), Z = C_{V-1}, s = logits - max, u in [0, 1)
    supplied by the caller;
  * the sliding-window threshold is tau_t = the mean of the last w token
    entropies including H_t, over the whole sequence (step boundaries play no
    part; truncated at the sequence start) -- the pages name the policy but do
    not write it out, and this is the window half of HSE used as the threshold
    at every position;
  * top-p keeps the smallest set of most probable tokens whose probability
    (at temperature T_t) reaches p, and keeps every token tied with the least
    probable one kept: token i stays iff the mass of the tokens with a
    strictly larger logit is below p * Z.  The kept tokens are renormalised and
    sampled inverse-CDF in vocabulary order, as above.  top_p = 1 keeps all.

Test infrastructure only (see the package docstring).
"""
import math
from dataclasses import dataclass, field

import numpy as np


THRESHOLDS = ("reset", "fixed", "window")


@dataclass
class ResetParams:
    tau0: float = 0.6
    t_low: float = 0.3
    t_high: float = 1.0
    w: int = 8
    threshold: str = "reset"        # one of THRESHOLDS
    top_p: float = 1.0              # in (0, 1]; 1 = no truncation


def token_entropy(logits: np.ndarray) -> float:
    """H = ln Z - (sum_i e^{s_i} s_i) / Z with s = l - max l, in FP64 (nats).
    A logit of -inf has probability 0 and adds nothing to the sum (the
    convention 0 log 0 = 0 of H = -sum p log p)."""
    l = np.asarray(logits, dtype=np.float64)
    s = l - np.max(l)
    e = np.exp(s)
    Z = np.sum(e)
    es = np.multiply(e, s, out=np.zeros_like(e), where=e > 0)
    return float(np.log(Z) - np.sum(es) / Z)


def nucleus_mask(logits: np.ndarray, T: float, top_p: float) -> np.ndarray:
    """Boolean [V]: the tokens top-p keeps at temperature T.  Token i stays iff
    sum of exp((l_j - max l) / T) over the tokens with l_j > l_i is below
    top_p * Z (so ties with the least probable kept token all stay)."""
    l = np.asarray(logits, dtype=np.float64)
    if top_p >= 1.0:
        return np.ones(l.shape, dtype=bool)
    e = np.exp((l - np.max(l)) / T)
    Z = float(np.sum(e))
    vals, inv = np.unique(l, return_inverse=True)       # ascending distinct logits
    group_mass = np.bincount(inv, weights=e, minlength=len(vals))
    # mass of the strictly larger logits, per distinct value
    above = np.concatenate([np.cumsum(group_mass[::-1])[::-1][1:], [0.0]])
    return (above < top_p * Z)[inv]


def sample_inverse_cdf(logits: np.ndarray, T: float, u: float, top_p: float = 1.0) -> int:
    """min{ i : C_i > u Z } for p_i proportional to exp((l_i - max l) / T),
    restricted to the nucleus_mask tokens (all of them when top_p = 1)."""
    l = np.asarray(logits, dtype=np.float64)
    e = np.exp((l - np.max(l)) / T) * nucleus_mask(l, T, top_p)
    C = np.cumsum(e)
    return int(np.argmax(C > u * C[-1]))


def acceptable_tokens(logits: np.ndarray, T: float, u: float, rel: float, keep=None) -> tuple[int, int]:
    """Range [lo, hi] of tokens that a sampler whose partial sums are accurate
    to rel * Z may return: lo samples at u - rel, hi at u + rel.  `keep`
    restricts the sample to a nucleus (boolean mask)."""
    l = np.asarray(logits, dtype=np.float64)
    e = np.exp((l - np.max(l)) / T)
    if keep is not None:
        e = e * keep
    C = np.cumsum(e)
    Z = C[-1]
    lo = int(np.argmax(C > max(u - rel, 0.0) * Z))
    hi_mask = C > min(u + rel, 1.0) * Z
    hi = int(np.argmax(hi_mask)) if hi_mask.any() else len(C) - 1
    return lo, hi


def nucleus_candidates(logits: np.ndarray, T: float, top_p: float, rel: float) -> list:
    """The nuclei a sampler whose masses are accurate to rel * Z may keep: the
    exact nucleus_mask, plus the one with its least probable logit group
    dropped when that group's `above` sum lies within rel * Z of top_p * Z, and
    the one with the next group added when that group's `above` sum does."""
    l = np.asarray(logits, dtype=np.float64)
    if top_p >= 1.0:
        return [np.ones(l.shape, dtype=bool)]
    e = np.exp((l - np.max(l)) / T)
    Z = float(np.sum(e))
    vals, inv = np.unique(l, return_inverse=True)
    group_mass = np.bincount(inv, weights=e, minlength=len(vals))
    above = np.concatenate([np.cumsum(group_mass[::-1])[::-1][1:], [0.0]])
    kept = above < top_p * Z                      # a suffix of the ascending groups
    out = [kept[inv]]
    g_last = int(np.argmax(kept))                 # least probable kept group
    if g_last + 1 < len(vals) and abs(above[g_last] - top_p * Z) <= rel * Z:
        k2 = kept.copy()
        k2[g_last] = False
        out.append(k2[inv])
    if g_last >= 1 and abs(above[g_last - 1] - top_p * Z) <= rel * Z:
        k3 = kept.copy()
        k3[g_last - 1] = True
        out.append(k3[inv])
    return out


@dataclass
class RowState:
    """Per-sequence ReSET state.  The oracle keeps the whole entropy history
    and forms every mean with an exactly rounded sum (math.fsum), so two means
    over the same set of entropies are bit-identical (at t < w the window is
    the whole history and equals the global mean)."""
    w: int
    t: int = 0                      # positions seen so far
    j: int = 0                      # 0-based position inside the current step
    hist: list = field(default_factory=list)   # H_0 .. H_{t-1}


@dataclass
class StepResult:
    H: float
    H_step: float
    H_bar: float
    tau: float
    T: float
    j: int
    H_win: float = 0.0


def reset_update(st: RowState, H: float, step_start: bool, p: ResetParams) -> StepResult:
    """Advance one row's state by one decode position and select T_t."""
    if st.t == 0 or step_start:
        st.j = 0
    st.hist.append(float(H))
    j = st.j
    win = st.hist[-p.w:]                          # last <= w entropies, may cross the step start
    H_win = math.fsum(win) / len(win)
    if j < p.w:
        H_step = H_win
    else:
        H_step = math.fsum(st.hist[-(j + 1):]) / (j + 1)   # positions 0..j of this step
    H_bar = math.fsum(st.hist) / (st.t + 1)
    if p.threshold == "fixed":                    # Eq. (1): one global threshold
        tau = p.tau0
    elif p.threshold == "window":                 # sliding-window threshold
        tau = H_win
    elif p.threshold == "reset":                  # SAT over the HSE estimate
        tau = p.tau0 if H_step <= H_bar else H_step
    else:
        raise ValueError(f"unknown threshold policy {p.threshold!r}")
    T = p.t_low if H < tau else p.t_high
    st.t += 1
    st.j += 1
    return StepResult(H=H, H_step=H_step, H_bar=H_bar, tau=tau, T=T, j=j, H_win=H_win)


def run_sequence(logits: np.ndarray, step_start: np.ndarray, u: np.ndarray, p: ResetParams):
    """Run the sampler over logits[steps, M, V] with flags step_start[steps, M]
    and uniforms u[steps, M].  Returns per-step, per-row StepResult lists and
    tokens [steps, M]."""
    steps, M, _ = logits.shape
    states = [RowState(w=p.w) for _ in range(M)]
    results = []
    tokens = np.zeros((steps, M), dtype=np.int64)
    for t in range(steps):
        row_res = []
        for r in range(M):
            H = token_entropy(logits[t, r])
            res = reset_update(states[r], H, bool(step_start[t, r]), p)
            tokens[t, r] = sample_inverse_cdf(logits[t, r], res.T, float(u[t, r]), p.top_p)
            row_res.append(res)
        results.append(row_res)
    return results, tokens


def temperature_is_ambiguous(res: StepResult, p: ResetParams, rel: float = 1e-4) -> bool:
    """True when H vs tau, or H_step vs H_bar, is within the comparison guard
    band, and the two sides of that comparison give different temperatures."""
    def pick_T(tau):
        return p.t_low if res.H < tau else p.t_high
    cands = {res.T}
    taus = [res.tau]
    if p.threshold == "reset" and abs(res.H_step - res.H_bar) <= rel * max(1.0, abs(res.H_bar)):
        taus = [p.tau0, res.H_step]
        cands.update(pick_T(tau) for tau in taus)
    for tau in taus:
        if abs(res.H - tau) <= rel * max(1.0, abs(tau)):
            cands.update({p.t_low, p.t_high})
    return len(cands) > 1
