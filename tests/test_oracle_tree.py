"""Pins of the oracle's greedy tree verification (reading R15)."""
import itertools

import numpy as np

from oracle import oracle


def test_chain_tree_is_the_linear_greedy_rule():
    # parents = i - 1: the tree is the drafted chain, so the result must be
    # the linear rule's (verify_row at T = 0 with the same N drafts)
    rng = np.random.default_rng(0)
    N, V = 6, 9
    for trial in range(200):
        tg = rng.normal(0, 1, (N + 1, V))
        am = tg.argmax(axis=1)
        tok = np.where(rng.random(N) < 0.7, am[:N], rng.integers(0, V, N)).astype(np.int32)
        d, toks, path = oracle.verify_tree_greedy_row(tg, tok, np.arange(N) - 1)
        lin = oracle.verify_row(tg, tg[:N], tok, np.zeros(N + 1), 0.0)
        assert d == lin.accepted_len
        assert toks == list(lin.out_tokens[:d + 1])
        assert path == list(range(d))


def test_the_lessons_six_node_tree():
    #        root
    #       /    \\
    #      a      b          a = node 0, b = node 1
    #     / \\    / \\
    #    c  d   e   f        c = 2, d = 3 (children of a); e = 4, f = 5 (of b)
    V = 10
    tok = np.array([1, 2, 3, 4, 5, 6])
    par = np.array([-1, -1, 0, 0, 1, 1])
    tg = np.zeros((7, V))
    tg[0, 2] = 5.0        # root slot: argmax 2 = token of b
    tg[1, 3] = 5.0        # slot after a: argmax 3 (c), but a is not accepted
    tg[2, 6] = 5.0        # slot after b: argmax 6 = token of f
    tg[6, 9] = 5.0        # slot after f: bonus 9
    d, toks, path = oracle.verify_tree_greedy_row(tg, tok, par)
    assert (d, toks, path) == (2, [2, 6, 9], [1, 5])
    # nothing accepted: the root's argmax alone
    tg2 = np.zeros((7, V))
    tg2[0, 8] = 1.0
    assert oracle.verify_tree_greedy_row(tg2, tok, par) == (0, [8], [])


def _brute(tg, tok, par):
    """Every root-to-node path, checked by the definition; the deepest
    accepted one, lowest end node on ties."""
    N = len(tok)
    am = tg.argmax(axis=1)
    best = None
    for end in range(N):
        path = []
        i = end
        while i >= 0:
            path.append(i)
            i = par[i]
        path = path[::-1]
        ok = all(tok[n] == am[0 if par[n] < 0 else par[n] + 1] for n in path)
        if ok and (best is None or len(path) > len(best)):
            best = path
    if best is None:
        return 0, [int(am[0])], []
    return len(best), [int(tok[n]) for n in best] + [int(am[best[-1] + 1])], best


def test_random_trees_against_path_enumeration():
    rng = np.random.default_rng(1)
    for trial in range(400):
        N = int(rng.integers(1, 12))
        V = int(rng.integers(2, 6))
        par = np.array([int(rng.integers(-1, i)) for i in range(N)])
        tg = rng.normal(0, 1, (N + 1, V))
        tok = rng.integers(0, V, N)
        assert oracle.verify_tree_greedy_row(tg, tok, par) == _brute(tg, tok, par)


def test_malformed_trees_are_error_rows():
    tg = np.zeros((4, 5))
    assert oracle.verify_tree_greedy_row(tg, np.array([0, 1, 2]), np.array([-1, 1, 0]))[0] == -1
    assert oracle.verify_tree_greedy_row(tg, np.array([0, 9, 2]), np.array([-1, 0, 1]))[0] == -1
    assert oracle.verify_tree_greedy_row(tg, np.array([0, 1, 2]), np.array([-2, 0, 1]))[0] == -1
    r = oracle.verify_tree_greedy(np.zeros((2, 4, 5)), np.array([[0, 1, 2], [0, 1, 2]]),
                                  np.array([[-1, 0, 1], [-1, 2, 0]]))
    # all-zero logits: every argmax is token 0, so row 0 accepts node 0 only
    assert list(r.accepted_len) == [1, -1] and (r.out_tokens[1] == -1).all()
    assert list(r.out_tokens[0]) == [0, 0, -1, -1] and list(r.accepted_nodes[0]) == [0, -1, -1]
