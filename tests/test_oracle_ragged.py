"""Pins of the oracle's adaptive-verification batch function
(``oracle.spec_verify_ragged``, reading R13: row b is the fixed-K rule on its
prefix of K_b drafted tokens, with u = uniforms[b, K_b])."""
import numpy as np
import pytest
from scipy.special import softmax

from oracle import oracle


def _batch(rng, B, K, V, T=1.0, scale=2.0):
    tg = rng.normal(0, scale, (B, K + 1, V))
    dr = tg[:, :K] + rng.normal(0, 0.5, (B, K, V))
    tokens = np.empty((B, K), np.int32)
    for b in range(B):
        for t in range(K):
            tokens[b, t] = rng.choice(V, p=softmax(dr[b, t] / T))
    unif = rng.random((B, K + 1))
    return tg, dr, tokens, unif, np.full(B, T)


def test_full_k_everywhere_is_the_fixed_k_rule():
    rng = np.random.default_rng(0)
    B, K, V = 12, 4, 9
    tg, dr, tok, un, T = _batch(rng, B, K, V)
    T[::4] = 0.0
    ref = oracle.spec_verify(tg, dr, tok, un, T)
    got = oracle.spec_verify_ragged(tg, dr, tok, un, T, np.full(B, K))
    np.testing.assert_array_equal(got.accepted_len, ref.accepted_len)
    np.testing.assert_array_equal(got.out_tokens, ref.out_tokens)
    np.testing.assert_array_equal(np.isnan(got.logp), np.isnan(ref.logp))
    np.testing.assert_allclose(got.logp[~np.isnan(ref.logp)], ref.logp[~np.isnan(ref.logp)], rtol=0, atol=0)


def test_no_drafted_tokens_draws_from_p0_with_u_at_column_zero():
    # K_b = 0: the row emits one token, the inverse CDF of p_0 at u = uniforms[b, 0]
    rng = np.random.default_rng(1)
    B, K, V = 40, 3, 11
    tg, dr, tok, un, T = _batch(rng, B, K, V, T=0.7)
    got = oracle.spec_verify_ragged(tg, dr, tok, un, T, np.zeros(B, np.int64))
    for b in range(B):
        p0 = softmax(tg[b, 0] / 0.7)                 # library softmax
        C = np.cumsum(p0)
        want = int(np.searchsorted(C, un[b, 0] * C[-1], side="right"))   # smallest i with C_i > uW
        assert got.accepted_len[b] == 0
        assert got.out_tokens[b, 0] == want
        assert (got.out_tokens[b, 1:] == -1).all()
        assert np.isnan(got.logp[b]).all() and np.isnan(got.logq[b]).all()


def test_prefix_rows_match_the_truncated_rule_and_pad():
    rng = np.random.default_rng(2)
    B, K, V = 16, 4, 7
    tg, dr, tok, un, T = _batch(rng, B, K, V)
    kb = rng.integers(0, K + 1, B)
    got = oracle.spec_verify_ragged(tg, dr, tok, un, T, kb)
    for b in range(B):
        k = int(kb[b])
        r = oracle.verify_row(tg[b, :k + 1], dr[b, :k], tok[b, :k], un[b, :k + 1], T[b])
        assert got.accepted_len[b] == r.accepted_len <= k
        np.testing.assert_array_equal(got.out_tokens[b, :k + 1], r.out_tokens)
        assert (got.out_tokens[b, k + 1:] == -1).all()
        np.testing.assert_array_equal(got.logp[b, :k], r.logp)
        assert np.isnan(got.logp[b, k:]).all()


def test_k_outside_the_padded_range_is_an_error_row():
    rng = np.random.default_rng(3)
    tg, dr, tok, un, T = _batch(rng, 3, 2, 5)
    got = oracle.spec_verify_ragged(tg, dr, tok, un, T, np.array([-1, 3, 2]))
    assert list(got.accepted_len[:2]) == [-1, -1]
    assert (got.out_tokens[:2] == -1).all()
    assert got.accepted_len[2] >= 0


@pytest.mark.parametrize("kb", [0, 1, 2, 4])
def test_expected_tokens_follow_the_closed_form_per_row_length(kb):
    # p = (0.9, 0.1), q = (0.7, 0.3) at every position: alpha = 0.8 exactly;
    # E[tokens] of a row verifying kb drafts is (1 - alpha^(kb+1)) / (1 - alpha)
    rng = np.random.default_rng(10 + kb)
    B, K = 6000, 4
    p = np.array([0.9, 0.1])
    q = np.array([0.7, 0.3])
    tg = np.broadcast_to(np.log(p), (B, K + 1, 2)).copy()
    dr = np.broadcast_to(np.log(q), (B, K, 2)).copy()
    tok = (rng.random((B, K)) < q[1]).astype(np.int32)      # x_t ~ q
    un = rng.random((B, K + 1))
    got = oracle.spec_verify_ragged(tg, dr, tok, un, np.ones(B), np.full(B, kb))
    tokens = got.accepted_len + 1
    mean, se = tokens.mean(), tokens.std() / np.sqrt(B)
    want = oracle.expected_tokens_closed_form(0.8, kb)
    assert abs(mean - want) < 4 * se + 1e-9
    assert (got.accepted_len <= kb).all()
