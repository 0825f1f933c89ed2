"""Pins for the CPU oracle: what the pages and the mathematics fix, not the
oracle's own formulas.

* closed forms of the softmax (two tokens = logistic, equal logits = 1/V,
  logits (0, ln 3) = (1/4, 3/4)) and its temperature;
* the inverse CDF reproduces its weights exactly on a fine u-grid and never
  picks a zero-weight token;
* the residual's mass equals the total-variation distance 1 - sum min(p, q);
* the exact output law of the rule, found by locating the oracle's own switch
  points in r_t and u, equals the law of plain sampling from p at every slot
  (the pages' distribution-preservation claim) and gives E[tokens] = 3.36 at
  alpha = 0.8, K = 4 as printed by the lesson;
* Monte Carlo over 10**6 oracle rows: chi-square and TV of every emitted slot
  against p;
* greedy rows equal argmax with the lowest index on ties;
* planted mistakes (scalar q in the residual, resampling from p on rejection,
  no bonus token, non-strict CDF comparison, T not applied to q) make these
  pins fail.
"""
from __future__ import annotations

import itertools
import math
import multiprocessing as mp
import os

import numpy as np
import pytest

from oracle import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- softmax pins

def test_log_softmax_two_tokens_is_logistic():
    z = np.array([0.3, -1.7])
    for T in (0.25, 1.0, 3.0):
        lp = oracle.log_softmax(z, T)
        p0 = 1.0 / (1.0 + math.exp((z[1] - z[0]) / T))
        assert abs(math.exp(lp[0]) - p0) < 1e-15
        assert abs(math.exp(lp[1]) - (1.0 - p0)) < 1e-15


def test_log_softmax_known_values_and_shift():
    lp = oracle.log_softmax(np.array([0.0, math.log(3.0)]), 1.0)
    assert np.allclose(np.exp(lp), [0.25, 0.75], atol=1e-15, rtol=0)
    # max shift keeps huge logits finite
    lp = oracle.log_softmax(np.array([1000.0, 1000.0 + math.log(3.0)]), 1.0)
    assert np.allclose(np.exp(lp), [0.25, 0.75], atol=1e-13, rtol=0)
    # equal logits -> uniform, for any temperature
    for T in (0.1, 1.0, 7.0):
        assert np.allclose(oracle.log_softmax(np.full(37, 2.5), T), -math.log(37), atol=1e-14)
    # temperature 2 on logits (0, 2 ln 3) is the same distribution as (0, ln 3)
    lp = oracle.log_softmax(np.array([0.0, 2 * math.log(3.0)]), 2.0)
    assert np.allclose(np.exp(lp), [0.25, 0.75], atol=1e-15, rtol=0)


def test_log_softmax_against_high_precision():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    rng = np.random.default_rng(5)
    z = rng.normal(0, 4, 200)
    z[7] = -np.inf
    T = 0.7
    lp = oracle.log_softmax(z, T)
    terms = [mpmath.e ** (mpmath.mpf(float(v)) / mpmath.mpf(T)) if np.isfinite(v) else mpmath.mpf(0)
             for v in z]
    S = mpmath.fsum(terms)
    for i in (0, 3, 50, 199):
        ref = mpmath.mpf(float(z[i])) / mpmath.mpf(T) - mpmath.log(S)
        assert abs(float(ref) - lp[i]) < 1e-12
    assert lp[7] == -np.inf


# ---------------------------------------------------------------- inverse CDF pins

def test_inverse_cdf_reproduces_weights_on_a_grid():
    w = np.array([0.0, 0.13, 0.0, 0.42, 0.05, 0.0, 0.4])
    N = 200_000
    u = (np.arange(N) + 0.5) / N
    counts = np.bincount([oracle.inverse_cdf(w, x) for x in u], minlength=len(w))
    assert np.all(counts[w == 0] == 0)
    assert np.allclose(counts / N, w / w.sum(), atol=2.0 / N)


def _check_zero_weight_edges():
    w = np.array([0.0, 0.0, 0.5, 0.0, 0.5, 0.0])
    assert oracle.inverse_cdf(w, 0.0) == 2
    assert oracle.inverse_cdf(w, 0.5) == 4          # C_2 = 0.5 is not > 0.5
    assert oracle.inverse_cdf(w, 1.0 - 2 ** -24) == 4
    assert oracle.inverse_cdf(w, 1.0) == 4          # rounding fallback: last positive weight


def test_inverse_cdf_never_picks_zero_weight_at_edges():
    _check_zero_weight_edges()


def test_cdf_margin_is_distance_to_nearest_boundary():
    w = np.array([0.25, 0.25, 0.5])
    assert abs(oracle.cdf_margin(w, 0.3) - 0.05) < 1e-15
    assert abs(oracle.cdf_margin(w, 0.9) - 0.1) < 1e-15


# ---------------------------------------------------------------- residual pins

def test_residual_mass_is_total_variation():
    rng = np.random.default_rng(1)
    for V in (2, 5, 1000):
        p = rng.dirichlet(np.ones(V))
        q = rng.dirichlet(np.ones(V))
        W = oracle.residual(p, q).sum()
        assert abs(W - (1.0 - np.minimum(p, q).sum())) < 1e-12
        assert abs(W - 0.5 * np.abs(p - q).sum()) < 1e-12
        assert abs((oracle.residual(p, q) / W).sum() - 1.0) < 1e-12


def test_residual_sat_slept_example():
    rows = _golden_rows("residual_example.txt")
    names = [r[0] for r in rows]
    p = np.array([float(r[1]) for r in rows])
    q = np.array([float(r[2]) for r in rows])
    w = oracle.residual(p, q)
    w = w / w.sum()
    # the token the draft over-proposed ("sat") drops to zero ...
    assert w[names.index("sat")] == 0.0
    # ... and the one it under-proposed ("slept") is boosted above its target probability
    assert w[names.index("slept")] > p[names.index("slept")]


# ---------------------------------------------------------------- exact law of the rule

def _bisect_threshold(pred):
    """sup{r in [0, 1): pred(r)} for a predicate true on [0, theta) and false after."""
    hi_r = 1.0 - 2.0 ** -53
    if pred(hi_r):
        return 1.0
    if not pred(0.0):
        return 0.0
    lo, hi = 0.0, hi_r
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if mid in (lo, hi):
            break
        if pred(mid):
            lo = mid
        else:
            hi = mid
    return hi


def _u_segments(f, a=0.0, b=1.0 - 2.0 ** -53, fa=None, fb=None, out=None):
    """Split [0, 1) into the pieces on which f (monotone step function of u) is constant."""
    top = out is None
    if top:
        out = []
        fa, fb = f(a), f(b)
    if fa == fb:
        out.append((fa, b - a))
    elif b - a < 1e-15:
        out.append((fa, 0.5 * (b - a)))
        out.append((fb, 0.5 * (b - a)))
    else:
        m = 0.5 * (a + b)
        fm = f(m)
        _u_segments(f, a, m, fa, fm, out)
        _u_segments(f, m, b, fm, fb, out)
    if top:
        # the last point b stands for [b, 1): fold that tiny remainder in
        return out
    return out


def exact_law(logP, logQ):
    """Law of (accepted_len, emitted tokens) of ``oracle.accept_and_sample`` when
    x_t ~ q_t and r_t, u ~ U(0, 1), computed from the oracle's own behaviour."""
    K, V = logQ.shape
    Q = np.exp(logQ)
    law = {}

    def run(x, rs, u):
        res = oracle.accept_and_sample(logP, logQ, np.array(x), np.array(list(rs) + [u]))
        n = int(res.accepted_len)
        return (n, tuple(int(v) for v in res.out_tokens[:n + 1]))

    def add(key, w):
        law[key] = law.get(key, 0.0) + w

    for x in itertools.product(range(V), repeat=K):
        weight = float(np.prod([Q[t, x[t]] for t in range(K)]))
        if weight == 0.0:
            continue
        rs = [0.5] * K
        survived = True
        for t in range(K):
            def accepted(r, t=t):
                rr = list(rs)
                rr[t] = r
                return run(x, rr, 0.5)[0] > t
            theta = _bisect_threshold(accepted)
            if theta < 1.0:
                rr = list(rs)
                rr[t] = 0.5 * (theta + 1.0)
                for key, length in _u_segments(lambda u: run(x, rr, u)):
                    add(key, weight * (1.0 - theta) * length)
            if theta == 0.0:
                survived = False
                break
            rs[t] = 0.5 * theta
            weight *= theta
        if survived:
            for key, length in _u_segments(lambda u: run(x, rs, u)):
                add(key, weight * length)
    return law


def slot_marginals(law, K, V):
    """For every slot s: P(slot s emitted) and P(token at slot s = v | emitted)."""
    emitted = np.zeros(K + 1)
    joint = np.zeros((K + 1, V))
    for (n, toks), w in law.items():
        for s in range(n + 1):
            emitted[s] += w
            joint[s, toks[s]] += w
    return emitted, joint / np.maximum(emitted, 1e-300)[:, None]


def _dists(rng, K, V, T=1.0, scale=1.0):
    tg = rng.normal(0, scale, (K + 1, V))
    dr = tg[:K] + rng.normal(0, scale, (K, V))
    logP = np.stack([oracle.log_softmax(tg[t], T) for t in range(K + 1)])
    logQ = np.stack([oracle.log_softmax(dr[t], T) for t in range(K)])
    return tg, dr, logP, logQ


@pytest.mark.parametrize("V,K,seed", [(2, 2, 0), (3, 2, 1), (4, 1, 2), (3, 3, 3)])
def test_exact_law_preserves_target_distribution(V, K, seed):
    rng = np.random.default_rng(seed)
    _, _, logP, logQ = _dists(rng, K, V)
    P = np.exp(logP)
    law = exact_law(logP, logQ)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    emitted, cond = slot_marginals(law, K, V)
    # the emitted token at every slot is distributed as p at that slot
    assert np.allclose(cond, P, atol=1e-12)
    # slot 1 is emitted with probability alpha_0 = sum min(p_0, q_0)
    Q = np.exp(logQ)
    assert abs(emitted[1] - np.minimum(P[0], Q[0]).sum()) < 1e-12


def test_temperature_applies_to_both_distributions():
    # the same logits verified at T = 2 must preserve softmax(target / 2) at each slot
    rng = np.random.default_rng(11)
    tg = rng.normal(0, 2, (3, 3))
    dr = tg[:2] + rng.normal(0, 2, (2, 3))
    T = 2.0
    logP = np.stack([oracle.log_softmax(tg[t], T) for t in range(3)])
    logQ = np.stack([oracle.log_softmax(dr[t], T) for t in range(2)])
    emitted, cond = slot_marginals(exact_law(logP, logQ), 2, 3)
    ref = np.exp(tg / T) / np.exp(tg / T).sum(axis=1, keepdims=True)
    assert np.allclose(cond, ref, atol=1e-12)


def _alpha08_dists(K):
    p = np.array([0.9, 0.1])
    q = np.array([0.7, 0.3])
    return np.log(np.tile(p, (K + 1, 1))), np.log(np.tile(q, (K, 1)))


def test_expected_tokens_matches_printed_value():
    alpha, K, printed, decimals = _golden_rows("expected_tokens.txt")[0]
    alpha, K, printed, decimals = float(alpha), int(K), float(printed), int(decimals)
    logP, logQ = _alpha08_dists(K)
    # sum of min(p, q) = 0.7 + 0.1 = 0.8 = alpha at every position
    assert abs(np.minimum(np.exp(logP[0]), np.exp(logQ[0])).sum() - alpha) < 1e-15
    law = exact_law(logP, logQ)
    E = sum(w * (n + 1) for (n, _), w in law.items())
    assert round(E, decimals) == printed
    assert abs(E - oracle.expected_tokens_closed_form(alpha, K)) < 1e-12
    # accepted_len is geometric: P(n = j) = alpha^j (1 - alpha), P(n = K) = alpha^K
    Pn = np.zeros(K + 1)
    for (n, _), w in law.items():
        Pn[n] += w
    ref = [alpha ** j * (1 - alpha) for j in range(K)] + [alpha ** K]
    assert np.allclose(Pn, ref, atol=1e-12)


def test_closed_form_extremes():
    assert oracle.expected_tokens_closed_form(0.0, 4) == 1.0
    assert oracle.expected_tokens_closed_form(1.0, 4) == 5.0
    assert abs(oracle.expected_tokens_closed_form(0.8, 4) - 3.3616) < 1e-12


# ---------------------------------------------------------------- planted mistakes

def _law_error(logP, logQ):
    K, V = logQ.shape
    emitted, cond = slot_marginals(exact_law(logP, logQ), K, V)
    return float(np.max(np.abs(cond - np.exp(logP))))


PLANTED = {
    # the code sketch's slip: subtract the scalar q(x_t) instead of the vector q
    "scalar_q_residual": "scalar",
    # resample from p on rejection
    "resample_from_p": "p",
    # no bonus token: stop after K accepted with argmax of nothing -> always token 0
    "no_bonus": "nobonus",
}


@pytest.mark.parametrize("mistake", sorted(PLANTED))
def test_planted_mistakes_break_preservation(monkeypatch, mistake):
    rng = np.random.default_rng(4)
    _, _, logP, logQ = _dists(rng, 2, 3)
    assert _law_error(logP, logQ) < 1e-12
    kind = PLANTED[mistake]
    if kind == "scalar":
        real = oracle.accept_and_sample

        def patched(lP, lQ, tokens, uniforms):
            # subtract the scalar q(x_t) like the sketch does
            orig = oracle.residual

            def scalar_res(p, q):
                t = next(i for i in range(len(tokens)) if np.allclose(q, np.exp(lQ[i])))
                return np.maximum(p - q[int(tokens[t])], 0.0)
            monkeypatch.setattr(oracle, "residual", scalar_res)
            try:
                return real(lP, lQ, tokens, uniforms)
            finally:
                monkeypatch.setattr(oracle, "residual", orig)
        monkeypatch.setattr(oracle, "accept_and_sample", patched)
    elif kind == "p":
        monkeypatch.setattr(oracle, "residual", lambda p, q: p.copy())
    else:
        real = oracle.accept_and_sample

        def patched(lP, lQ, tokens, uniforms):
            res = real(lP, lQ, tokens, uniforms)
            if res.accepted_len == len(tokens):
                res.out_tokens[-1] = 0
            return res
        monkeypatch.setattr(oracle, "accept_and_sample", patched)
    assert _law_error(logP, logQ) > 1e-3


def test_planted_non_strict_cdf_picks_zero_weight(monkeypatch):
    def non_strict(w, u):
        C = np.cumsum(w)
        return int(np.nonzero(C >= u * C[-1])[0][0])
    monkeypatch.setattr(oracle, "inverse_cdf", non_strict)
    with pytest.raises(AssertionError):
        _check_zero_weight_edges()


def test_planted_temperature_on_target_only_breaks_preservation(monkeypatch):
    rng = np.random.default_rng(11)
    tg = rng.normal(0, 2, (3, 3))
    dr = tg[:2] + rng.normal(0, 2, (2, 3))
    logP = np.stack([oracle.log_softmax(tg[t], 2.0) for t in range(3)])
    logQ_wrong = np.stack([oracle.log_softmax(dr[t], 1.0) for t in range(2)])
    # tokens drafted at T = 2 but q evaluated at T = 1
    logQ_true = np.stack([oracle.log_softmax(dr[t], 2.0) for t in range(2)])
    K, V = 2, 3
    real = oracle.accept_and_sample
    monkeypatch.setattr(oracle, "accept_and_sample",
                        lambda lP, lQ, tk, un: real(lP, logQ_wrong, tk, un))
    emitted, cond = slot_marginals(exact_law(logP, logQ_true), K, V)
    assert np.max(np.abs(cond - np.exp(logP))) > 1e-3


# ---------------------------------------------------------------- Monte Carlo pins

def _mc_worker(args):
    logP, logQ, n, seed = args
    from oracle import oracle as orc
    rng = np.random.default_rng(seed)
    K, V = logQ.shape
    Q = np.exp(logQ)
    counts = np.zeros((K + 1, V), np.int64)
    tokens_total = 0
    for _ in range(n):
        x = np.array([rng.choice(V, p=Q[t]) for t in range(K)])
        res = orc.accept_and_sample(logP, logQ, x, rng.random(K + 1))
        nacc = int(res.accepted_len)
        tokens_total += nacc + 1
        for s in range(nacc + 1):
            counts[s, res.out_tokens[s]] += 1
    return counts, tokens_total


def _mc(logP, logQ, n, seed, workers=8):
    per = n // workers
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers) as pool:
        parts = pool.map(_mc_worker, [(logP, logQ, per, seed * 1000 + i) for i in range(workers)])
    counts = sum(p[0] for p in parts)
    return counts, sum(p[1] for p in parts), per * workers


@pytest.mark.slow
def test_monte_carlo_chi_square_every_slot():
    scipy_stats = pytest.importorskip("scipy.stats")
    samples, tv_bar, _ = _golden_rows("distribution_check.txt")[0]
    tv_bar = float(tv_bar)
    rng = np.random.default_rng(21)
    K, V = 3, 8
    _, _, logP, logQ = _dists(rng, K, V, T=1.0, scale=1.2)
    counts, _, n = _mc(logP, logQ, 1_000_000, seed=7)
    P = np.exp(logP)
    assert counts[0].sum() == n
    for s in range(K + 1):
        c = counts[s]
        m = c.sum()
        assert m > 10_000
        stat, pval = scipy_stats.chisquare(c, m * P[s])
        assert pval > 1e-3, (s, pval)
        assert 0.5 * np.abs(c / m - P[s]).sum() < tv_bar


@pytest.mark.slow
def test_monte_carlo_expected_tokens_alpha_08():
    logP, logQ = _alpha08_dists(4)
    _, total, n = _mc(logP, logQ, 200_000, seed=3)
    mean = total / n
    E = 3.3616
    # var of tokens for the truncated geometric with alpha = 0.8, K = 4
    ps = np.array([0.8 ** j * 0.2 for j in range(4)] + [0.8 ** 4])
    vals = np.arange(1, 6)
    var = (ps * vals ** 2).sum() - E ** 2
    assert abs(mean - E) < 4 * math.sqrt(var / n)


# ---------------------------------------------------------------- rule special cases

def test_q_equal_p_accepts_everything():
    rng = np.random.default_rng(2)
    K, V = 4, 50
    tg = rng.normal(0, 2, (K + 1, V))
    for r in (0.0, 0.5, 1.0 - 2 ** -24):
        res = oracle.verify_row(tg, tg[:K], rng.integers(0, V, K), np.full(K + 1, r), 1.0)
        assert res.accepted_len == K
        assert res.mode == "bonus"


def test_greedy_rule_and_lowest_index_ties():
    V = 6
    tg = np.array([[0, 5, 5, 1, 0, 0],      # argmax 1 (tie with 2 -> lowest)
                   [9, 0, 0, 0, 0, 9],      # argmax 0
                   [0, 0, 0, 0, 3, 0],      # argmax 4
                   [1, 1, 1, 1, 1, 1]],     # bonus: argmax 0
                  float)
    garbage = np.full((3, V), np.nan)       # greedy rows never read the draft
    res = oracle.verify_row(tg, garbage, np.array([1, 0, 4]), np.full(4, np.nan), 0.0)
    assert res.accepted_len == 3 and list(res.out_tokens) == [1, 0, 4, 0]
    res = oracle.verify_row(tg, garbage, np.array([1, 5, 4]), np.zeros(4), 0.0)
    assert res.accepted_len == 1 and list(res.out_tokens) == [1, 0, -1, -1]
    res = oracle.verify_row(tg, garbage, np.array([2, 0, 4]), np.zeros(4), 0.0)
    assert res.accepted_len == 0 and list(res.out_tokens) == [1, -1, -1, -1]


def test_greedy_matches_brute_force_argmax():
    rng = np.random.default_rng(9)
    for _ in range(50):
        V, K = 11, 3
        tg = rng.integers(-3, 3, (K + 1, V)).astype(float)   # many ties
        x = rng.integers(0, V, K)
        res = oracle.verify_row(tg, np.zeros((K, V)), x, np.zeros(K + 1), 0.0)
        # brute force: scan left to right keeping the first maximum
        def first_max(row):
            best, bi = -np.inf, -1
            for i, v in enumerate(row):
                if v > best:
                    best, bi = v, i
            return bi
        n = 0
        while n < K and first_max(tg[n]) == x[n]:
            n += 1
        assert res.accepted_len == n
        assert res.out_tokens[n] == first_max(tg[n])


def test_error_rows():
    K, V = 2, 5
    tg = np.zeros((K + 1, V))
    for T in (-1.0, np.nan, np.inf, 1e-39):
        res = oracle.verify_row(tg, tg[:K], np.array([0, 1]), np.zeros(K + 1), T)
        assert res.accepted_len == -1 and (res.out_tokens == -1).all()
    for bad in ([0, 5], [-1, 0]):
        res = oracle.verify_row(tg, tg[:K], np.array(bad), np.zeros(K + 1), 1.0)
        assert res.accepted_len == -1
    allinf = np.full((K + 1, V), -np.inf)
    assert oracle.verify_row(allinf, tg[:K], np.array([0, 1]), np.zeros(K + 1), 1.0).accepted_len == -1


def test_neg_inf_logit_token_is_always_rejected():
    K, V = 1, 4
    tg = np.array([[0.0, -np.inf, 1.0, 2.0], [0.0, 0.0, 0.0, 0.0]])
    dr = np.array([[0.0, 3.0, 1.0, 2.0]])
    for r in (0.0, 0.3):
        res = oracle.verify_row(tg, dr, np.array([1]), np.array([r, 0.5]), 1.0)
        assert res.accepted_len == 0 and res.out_tokens[0] != 1


def test_batch_wrapper_decodes_bf16():
    # bf16 bit patterns of 1.0 (0x3F80) and 2.0 (0x4000)
    raw_t = np.array([[[0x3F80, 0x4000], [0x4000, 0x3F80]]], np.uint16)
    raw_d = np.array([[[0x3F80, 0x4000]]], np.uint16)
    out = oracle.spec_verify(raw_t, raw_d, np.array([[1]]), np.array([[0.0, 0.5]], np.float32),
                             np.array([0.0], np.float32), dtype="bf16")
    assert out.accepted_len[0] == 1 and list(out.out_tokens[0]) == [1, 0]
