"""Pins of the oracle's plug step (reading R14)."""
import numpy as np

from oracle import oracle


def test_worked_example():
    # row 0: 2 accepted + replacement at length 3; row 1: error row;
    # row 2: 0 accepted (1 token) at length 0; row 3: bonus (K+1 = 3 tokens)
    # at length 6 of 8 -> the last one does not fit
    acc = np.array([2, -1, 0, 2])
    out = np.array([[11, 12, 13], [-1, -1, -1], [21, -1, -1], [31, 32, 33]])
    tok = np.full((4, 8), 7)
    L = np.array([3, 5, 0, 6])
    r = oracle.plug(acc, out, tok, L, last_token=np.array([1, 2, 3, 4]))
    np.testing.assert_array_equal(r.tokens[0], [7, 7, 7, 11, 12, 13, 7, 7])
    np.testing.assert_array_equal(r.tokens[1], [7] * 8)
    np.testing.assert_array_equal(r.tokens[2], [21, 7, 7, 7, 7, 7, 7, 7])
    np.testing.assert_array_equal(r.tokens[3], [7, 7, 7, 7, 7, 7, 31, 32])
    np.testing.assert_array_equal(r.seq_len, [6, 5, 1, 8])
    np.testing.assert_array_equal(r.last_token, [13, 2, 21, 33])
    np.testing.assert_array_equal(r.clipped, [False, False, False, True])


def test_invariants_on_random_states():
    rng = np.random.default_rng(0)
    B, K, max_len = 50, 5, 40
    acc = rng.integers(-1, K + 1, B)
    out = np.full((B, K + 1), -1)
    for b in range(B):
        if acc[b] >= 0:
            out[b, :acc[b] + 1] = rng.integers(0, 1000, acc[b] + 1)
    tok = rng.integers(0, 1000, (B, max_len))
    L = rng.integers(0, max_len + 1, B)
    r = oracle.plug(acc, out, tok, L)
    for b in range(B):
        n, l0 = int(acc[b]), int(L[b])
        assert (r.tokens[b, :l0] == tok[b, :l0]).all()            # the prefix is untouched
        if n < 0:
            assert r.seq_len[b] == l0 and (r.tokens[b] == tok[b]).all()
            continue
        fit = min(n + 1, max_len - l0)
        assert r.seq_len[b] == l0 + fit
        assert (r.tokens[b, l0:l0 + fit] == out[b, :fit]).all()
        assert (r.tokens[b, l0 + fit:] == tok[b, l0 + fit:]).all()
        assert r.clipped[b] == (fit < n + 1)
        assert r.last_token[b] == out[b, n]


def test_length_outside_the_buffer_leaves_the_row():
    acc = np.array([1, 1])
    out = np.array([[5, 6], [7, 8]])
    tok = np.zeros((2, 4), np.int32)
    r = oracle.plug(acc, out, tok, np.array([-1, 5]))
    np.testing.assert_array_equal(r.seq_len, [-1, 5])
    assert (r.tokens == 0).all() and not r.clipped.any()


def test_length_past_the_padded_row_leaves_the_row():
    # accepted_len above K is not an output of the verify step: nothing moves
    acc = np.array([2, 3, 1])
    out = np.array([[5, 6, 7], [8, 9, 10], [11, 12, -1]])
    tok = np.zeros((3, 6), np.int32)
    r = oracle.plug(acc, out, tok, np.array([0, 0, 0]), last_token=np.array([-5, -5, -5]))
    np.testing.assert_array_equal(r.seq_len, [3, 0, 2])
    np.testing.assert_array_equal(r.tokens[1], [0] * 6)
    np.testing.assert_array_equal(r.last_token, [7, -5, 12])
