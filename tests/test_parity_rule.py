"""The comparison rule that the GPU parity tests and the bench's parity block
apply (oracle/parity.py), checked on planted differences: every kind of
mismatch the rule must catch is caught, and only mismatches on rows the
oracle marks ambiguous are let through (counted)."""
from __future__ import annotations

import dataclasses

import numpy as np

from oracle import oracle
from oracle.parity import LOGPROB_ATOL, MARGIN, check_structure, compare
from speculative_decoding_verification_25_gb300 import synth


def _batch():
    """Eight tiny rows through the oracle: six tempered, two greedy."""
    ws = [synth.make("tiny_stochastic", seed=s) for s in range(6)]
    ws += [synth.make("tiny_greedy", seed=s) for s in range(2)]
    cat = lambda f: np.concatenate([getattr(w, f) for w in ws])
    tgt, dft, tok, uni, temp = (cat("target"), cat("draft"), cat("draft_tokens"),
                                cat("uniforms"), cat("temperature"))
    ref = oracle.spec_verify(tgt, dft, tok, uni, temp, dtype=ws[0].dtype)
    return ref, tok, temp, ws[0].V


def _gpu_like(ref):
    """Outputs in the GPU's types, equal to the oracle's."""
    return (ref.accepted_len.astype(np.int32).copy(), ref.out_tokens.astype(np.int32).copy(),
            ref.logp.astype(np.float32), ref.logq.astype(np.float32))


def _other_token(t, V):
    return (int(t) + 1) % V


def test_identical_outputs_pass():
    ref, tok, temp, V = _batch()
    acc, out, lp, lq = _gpu_like(ref)
    rep = compare(ref, acc, out, lp, lq, temp)
    assert rep.rows == 8 and rep.greedy_rows == 2 and rep.stochastic_rows == 6
    assert rep.mismatched_rows == 0 and not rep.failures
    assert not check_structure(acc, out, tok, V)


def test_greedy_row_mismatch_fails():
    ref, tok, temp, V = _batch()
    acc, out, lp, lq = _gpu_like(ref)
    g = 6                                   # a greedy row
    n = acc[g]
    out[g, n] = _other_token(out[g, n], V)
    rep = compare(ref, acc, out, lp, lq, temp)
    assert len(rep.failures) == 1 and rep.failures[0][0] == g


def test_unambiguous_stochastic_mismatch_fails():
    ref, tok, temp, V = _batch()
    acc, out, lp, lq = _gpu_like(ref)
    ref = dataclasses.replace(ref, cdf_margin=np.full_like(ref.cdf_margin, 1.0),
                              ratio_margin=np.full_like(ref.ratio_margin, 1.0))
    b = 0
    out[b, acc[b]] = _other_token(out[b, acc[b]], V)
    rep = compare(ref, acc, out, lp, lq, temp)
    assert rep.mismatched_rows == 1 and rep.ambiguous_rows == 0
    assert len(rep.failures) == 1 and "unambiguous" in rep.failures[0][1]


def test_ambiguous_mismatch_is_counted_not_failed():
    ref, tok, temp, V = _batch()
    acc, out, lp, lq = _gpu_like(ref)
    cm = np.full_like(ref.cdf_margin, 1.0)
    rm = np.full_like(ref.ratio_margin, 1.0)
    cm[1] = MARGIN / 2                      # u near a CDF boundary
    rm[2, 0] = MARGIN / 2                   # r_0 near p/q: a decided position
    ref = dataclasses.replace(ref, cdf_margin=cm, ratio_margin=rm)
    for b in (1, 2):
        out[b, acc[b]] = _other_token(out[b, acc[b]], V)
    rep = compare(ref, acc, out, lp, lq, temp)
    assert rep.ambiguous_rows == 2 and rep.mismatched_rows == 2 and not rep.failures


def test_ratio_margin_after_the_decided_positions_does_not_count():
    """Only positions 0..n decide the row: a small margin past them is not
    ambiguity."""
    ref, tok, temp, V = _batch()
    acc, out, lp, lq = _gpu_like(ref)
    b = int(np.argmin(np.where(temp[:6] > 0, acc[:6], 99)))   # a tempered row with the fewest accepted
    K = ref.ratio_margin.shape[1]
    assert acc[b] + 1 < K, "the batch should hold a tempered row rejected before its last position"
    rm = np.full_like(ref.ratio_margin, 1.0)
    rm[b, acc[b] + 1:] = MARGIN / 2
    ref = dataclasses.replace(ref, cdf_margin=np.full_like(ref.cdf_margin, 1.0), ratio_margin=rm)
    out[b, acc[b]] = _other_token(out[b, acc[b]], V)
    rep = compare(ref, acc, out, lp, lq, temp)
    assert rep.ambiguous_rows == 0 and len(rep.failures) == 1


def test_logprob_tolerance_and_special_values():
    ref, tok, temp, V = _batch()
    acc, out, lp, lq = _gpu_like(ref)
    lp = lp.astype(np.float64)
    lp[0, 0] += 3 * LOGPROB_ATOL
    rep = compare(ref, acc, out, lp, lq, temp)
    assert len(rep.failures) == 1 and "log-prob" in rep.failures[0][1]
    # equal -inf on both sides is exact; NaN on one side only is an infinite error
    ref2 = dataclasses.replace(ref, logp=ref.logp.copy())
    ref2.logp[0, 0] = -np.inf
    lp2 = ref2.logp.astype(np.float32)
    assert not compare(ref2, acc, out, lp2, lq, temp).failures
    lp3 = lp2.copy()
    lp3[0, 1] = np.nan
    rep3 = compare(ref2, acc, out, lp3, lq, temp)
    assert rep3.failures and rep3.max_logprob_err == np.inf


def test_rows_mapping():
    """rows[i] names the GPU row that oracle row i is compared with."""
    ref, tok, temp, V = _batch()
    acc, out, lp, lq = _gpu_like(ref)
    perm = np.array([3, 0, 1, 2, 4, 5, 7, 6])      # oracle row i sits at GPU row perm[i]

    def place(x):
        y = np.empty_like(x)
        y[perm] = x
        return y

    args = [place(x) for x in (acc, out, lp, lq, temp)]
    rep = compare(ref, *args, rows=perm)
    assert rep.rows == 8 and not rep.failures and rep.mismatched_rows == 0
    # the identity mapping on permuted outputs is caught
    assert compare(ref, *args).failures


def test_structure_checks():
    ref, tok, temp, V = _batch()
    acc, out, lp, lq = _gpu_like(ref)
    K = out.shape[1] - 1
    cases = []
    a, o = acc.copy(), out.copy()
    a[0] = -1                                   # an error row must carry -1 tokens only
    cases.append((a, o, "error row with tokens"))
    a, o = acc.copy(), out.copy()
    a[1] = K + 1
    cases.append((a, o, "accepted_len"))
    a, o = acc.copy(), out.copy()
    a[2] = max(a[2], 1)
    o[2, :a[2]] = tok[2, :a[2]]
    o[2, 0] = _other_token(tok[2, 0], V)
    cases.append((a, o, "accepted prefix"))
    a, o = acc.copy(), out.copy()
    o[3, a[3]] = V
    cases.append((a, o, "out of range"))
    a, o = acc.copy(), out.copy()
    if a[4] < K:
        o[4, K] = 0
        cases.append((a, o, "padding"))
    for a, o, what in cases:
        bad = check_structure(a, o, tok, V)
        assert bad and any(what in msg for _, msg in bad), (what, bad)
