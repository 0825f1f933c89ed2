"""The seeded input generator: determinism, shapes, ranges and recipe."""
import numpy as np
import pytest

from speculative_decoding_verification_25_gb300 import synth


def test_same_seed_same_bytes_and_subsets_match():
    a = synth.make("greedy_batch", seed=3, rows=[0, 5, 31])
    b = synth.make("greedy_batch", seed=3, rows=[5])
    assert np.array_equal(a.target[1], b.target[0])
    assert np.array_equal(a.draft[1], b.draft[0])
    assert np.array_equal(a.draft_tokens[1], b.draft_tokens[0])
    c = synth.make("greedy_batch", seed=4, rows=[5])
    assert not np.array_equal(c.target[0], b.target[0])


def test_pool_build_equals_serial_build():
    a = synth.make("tiny_stochastic", seed=0)
    b = synth.make("greedy_batch", seed=1, rows=range(4), workers=2)
    c = synth.make("greedy_batch", seed=1, rows=range(4), workers=1)
    assert np.array_equal(b.target, c.target) and np.array_equal(b.draft_tokens, c.draft_tokens)
    assert a.target.dtype == np.float32 and b.target.dtype == np.uint16


@pytest.mark.parametrize("name", synth.ORDER + ["tiny_greedy"])
def test_shapes_ranges_and_temperatures(name):
    cfg = synth.WORKLOADS[name]
    rows = [0, 1, 2, 10] if cfg["B"] > 10 else list(range(cfg["B"]))
    w = synth.make(name, seed=0, rows=rows)
    B, K, V = len(rows), cfg["K"], cfg["V"]
    assert w.target.shape == (B, K + 1, V) and w.draft.shape == (B, K, V)
    assert w.draft_tokens.shape == (B, K) and w.uniforms.shape == (B, K + 1)
    assert (w.draft_tokens >= 0).all() and (w.draft_tokens < V).all()
    assert (w.uniforms >= 0).all() and (w.uniforms < 1).all()
    T = w.temperature
    if name in ("greedy_batch", "tiny_greedy"):
        assert (T == 0).all()
    if name == "long_draft_mixed_t":
        assert T[0] == 0 and T[3] == 0 and 0.3 <= T[1] <= 1.5
    if name == "large_vocab_stress":
        assert T[0] == np.float32(0.7) and T[1] == 0


def test_greedy_tokens_are_draft_argmax():
    w = synth.make("greedy_batch", seed=0, rows=[0, 1])
    d = (w.draft.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(w.draft_tokens, np.argmax(d, axis=-1))


def test_planted_peak_present():
    w = synth.make("greedy_batch", seed=0, rows=[0])
    t = (w.target.astype(np.uint32) << 16).view(np.float32)
    # one +8 peak on N(0, 3): the row maximum sits well above the bulk
    assert (t.max(axis=-1) > 8.0).all()


def test_drafted_tokens_follow_q_in_law():
    # Gumbel-max sampling over many seeds on a 4-token row reproduces softmax(d / T)
    counts = np.zeros(4)
    d = np.array([0.0, 1.0, -0.5, 0.3])
    for s in range(4000):
        wl = synth.custom(np.zeros((1, 2, 4)), d[None, None], [[0]], [[0.5, 0.5]], [1.0])
        U = synth._rng(s, 99, 0, 3).random(4)
        counts[np.argmax(d + -np.log(-np.log(U)))] += 1
    p = np.exp(d) / np.exp(d).sum()
    assert np.abs(counts / counts.sum() - p).max() < 0.03


def test_ragged_workload_rows_and_lengths():
    from speculative_decoding_verification_25_gb300 import synth
    w = synth.make("llama3_ragged", seed=0, rows=[0, 5, 9])
    assert w.k_per_row is not None and w.k_per_row.dtype == np.int32
    assert ((w.k_per_row >= 0) & (w.k_per_row <= w.K)).all()
    # the same rows rebuilt alone give the same lengths and values
    w2 = synth.make("llama3_ragged", seed=0, rows=[9])
    assert w2.k_per_row[0] == w.k_per_row[2]
    np.testing.assert_array_equal(w2.target[0], w.target[2])
    full = synth.make("llama3_ragged", seed=1, rows=range(64)).k_per_row
    assert set(full.tolist()) == set(range(w.K + 1))   # every length occurs
    assert synth.make("llama3_stochastic", seed=0, rows=[0]).k_per_row is None


def test_tree_workload_shape_and_parents():
    from speculative_decoding_verification_25_gb300 import synth
    np.testing.assert_array_equal(synth.tree_parents((2, 1)), [-1, -1, 0, 1])
    w = synth.make("llama3_tree", seed=0, rows=[0, 3])
    N = w.K
    assert w.parents.shape == (2, N) and w.target.shape == (2, N + 1, w.V)
    assert all(-1 <= w.parents[0, i] < i for i in range(N))
    assert ((w.draft_tokens >= 0) & (w.draft_tokens < w.V)).all()
    assert (w.temperature == 0).all()
    w2 = synth.make("llama3_tree", seed=0, rows=[3])
    np.testing.assert_array_equal(w2.draft_tokens[0], w.draft_tokens[1])
