"""CUDA path vs the CPU oracle, through the C ABI, on the five synthetic
workloads at full size (the launch configuration the benchmark times) and on
small shapes that cover the edge cases."""
from __future__ import annotations

import numpy as np
import pytest

from speculative_decoding_verification_25_gb300 import synth

from _parity import check_structure, compare
from gpu_util import device_tensors, run_gpu, run_oracle, run_oracle_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from speculative_decoding_verification_25_gb300 import build as b
    b.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield


def _assert_parity(rep, max_mismatch):
    assert not rep.failures, rep.failures[:5]
    assert rep.mismatched_rows <= max_mismatch, rep


# ---------------------------------------------------------------- tiny workloads

@pytest.mark.parametrize("name", ["tiny_stochastic", "tiny_greedy"])
def test_tiny_workload_matches_oracle(name):
    total = None
    for seed in range(24):
        w = synth.make(name, seed=seed)
        g = run_gpu(w)
        ref = run_oracle(w, workers=1)
        assert not check_structure(g["accepted"], g["out_tokens"], w.draft_tokens, w.V)
        rep = compare(ref, g["accepted"], g["out_tokens"], g["logp"], g["logq"], w.temperature)
        total = rep if total is None else total.merge(rep)
    _assert_parity(total, 0)


# ---------------------------------------------------------------- full-size workloads

@pytest.mark.parametrize("seed", [0, 1])
def test_greedy_batch_full_size_bit_exact(seed):
    w = synth.make("greedy_batch", seed=seed, workers=synth.default_workers())
    g = run_gpu(w)
    ref = run_oracle(w)
    assert not check_structure(g["accepted"], g["out_tokens"], w.draft_tokens, w.V)
    rep = compare(ref, g["accepted"], g["out_tokens"], g["logp"], g["logq"], w.temperature)
    assert rep.greedy_rows == w.B
    _assert_parity(rep, 0)
    # greedy rows report no log-probabilities
    assert np.isnan(g["logp"]).all() and np.isnan(g["logq"]).all()


def test_llama3_stochastic_full_size():
    """B=64, K=4, V=128256 bf16 at 8 seeds: every row checked."""
    total = None
    for seed in range(8):
        w = synth.make("llama3_stochastic", seed=seed, workers=synth.default_workers())
        g = run_gpu(w)
        ref = run_oracle(w)
        assert not check_structure(g["accepted"], g["out_tokens"], w.draft_tokens, w.V)
        rep = compare(ref, g["accepted"], g["out_tokens"], g["logp"], g["logq"], w.temperature)
        total = rep if total is None else total.merge(rep)
    print("llama3_stochastic parity:", total)
    assert total.stochastic_rows == 8 * 64
    _assert_parity(total, int(0.001 * total.rows))


@pytest.mark.parametrize("seed", [0, 1])
def test_long_draft_mixed_t_full_size(seed):
    """B=256, K=8, V=152064 fp32 (26 greedy rows, T ~ U(0.3, 1.5) on the
    others): every row against the oracle."""
    w = synth.make("long_draft_mixed_t", seed=seed, workers=synth.default_workers())
    g = run_gpu(w)
    assert not check_structure(g["accepted"], g["out_tokens"], w.draft_tokens, w.V)
    temperature = w.temperature
    del w
    ref = run_oracle_workload("long_draft_mixed_t", seed, 256)
    rep = compare(ref, g["accepted"], g["out_tokens"], g["logp"], g["logq"], temperature)
    print(f"long_draft_mixed_t seed {seed} parity:", rep)
    assert rep.rows == 256 and rep.greedy_rows == 26 and rep.stochastic_rows == 230
    _assert_parity(rep, 0)


@pytest.mark.parametrize("seed", [0, 1])
def test_large_vocab_stress_full_size(seed):
    """B=512, K=10, V=262144 bf16 (5.6 GB of logits; odd rows greedy, even
    rows T = 0.7): every row against the oracle."""
    w = synth.make("large_vocab_stress", seed=seed, workers=synth.default_workers())
    g = run_gpu(w)
    assert not check_structure(g["accepted"], g["out_tokens"], w.draft_tokens, w.V)
    temperature = w.temperature
    del w
    ref = run_oracle_workload("large_vocab_stress", seed, 512)
    rep = compare(ref, g["accepted"], g["out_tokens"], g["logp"], g["logq"], temperature)
    print(f"large_vocab_stress seed {seed} parity:", rep)
    assert rep.rows == 512 and rep.greedy_rows == 256 and rep.stochastic_rows == 256
    _assert_parity(rep, 0)


def test_shapes_change_on_one_workspace():
    """Calls of different shapes share one (never initialised) workspace."""
    import torch
    from speculative_decoding_verification_25_gb300 import api
    ws = torch.full((64 << 20,), 0xAB, dtype=torch.uint8, device="cuda:0")   # garbage
    for name, rows in (("greedy_batch", range(7)), ("llama3_stochastic", range(12)),
                       ("tiny_stochastic", None), ("long_draft_mixed_t", range(5)),
                       ("llama3_stochastic", range(3)), ("llama3_ragged", range(9))):
        w = synth.make(name, seed=2, rows=rows)
        d = device_tensors(w)
        r = api.spec_verify(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                            d["temperature"], k_per_row=d.get("k_per_row"), want_logprobs=True,
                            workspace=ws)
        torch.cuda.synchronize()
        ref = run_oracle(w, workers=1)
        rep = compare(ref, r.accepted_len.cpu().numpy(), r.out_tokens.cpu().numpy(),
                      r.logp.cpu().numpy(), r.logq.cpu().numpy(), w.temperature)
        _assert_parity(rep, 0)


@pytest.mark.parametrize("name,rows", [("llama3_stochastic", range(8)), ("llama3_ragged", range(12)),
                                       ("tiny_stochastic", None), ("greedy_batch", range(5))])
def test_row_stats_alone_leaves_the_partials_the_step_folds(name, rows):
    """spec_verify_row_stats writes, for every row the step reads, the same
    tile partials (bit for bit) as the first launch of spec_verify."""
    import torch
    from speculative_decoding_verification_25_gb300 import _native as N
    w = synth.make(name, seed=4, rows=rows)
    d = device_tensors(w)
    dt = N.SV_BF16 if w.dtype == "bf16" else N.SV_F32
    B, K, V = w.B, w.K, w.V
    nb = N.spec_verify_workspace_bytes(B, K, V, dt)
    sh = torch.cuda.current_stream().cuda_stream
    kp = d["k_per_row"].data_ptr() if "k_per_row" in d else 0
    ws1 = torch.full((nb,), 0x5A, dtype=torch.uint8, device="cuda:0")
    ws2 = torch.full((nb,), 0xA5, dtype=torch.uint8, device="cuda:0")
    assert N.spec_verify_row_stats_raw(d["target"].data_ptr(), d["draft"].data_ptr(), dt,
                                       d["temperature"].data_ptr(), kp, B, K, V, ws1.data_ptr(),
                                       nb, sh) == N.SV_OK
    acc = torch.empty(B, dtype=torch.int32, device="cuda:0")
    out = torch.empty(B, K + 1, dtype=torch.int32, device="cuda:0")
    args = (d["draft_tokens"].data_ptr(), d["uniforms"].data_ptr(), d["temperature"].data_ptr())
    if kp:
        st = N.spec_verify_ragged_raw(d["target"].data_ptr(), d["draft"].data_ptr(), dt, *args, kp,
                                      B, K, V, acc.data_ptr(), out.data_ptr(), None, None,
                                      ws2.data_ptr(), nb, sh)
    else:
        st = N.spec_verify_raw(d["target"].data_ptr(), d["draft"].data_ptr(), dt, *args, B, K, V,
                               acc.data_ptr(), out.data_ptr(), None, None, ws2.data_ptr(), nb, sh)
    assert st == N.SV_OK
    torch.cuda.synchronize()
    a, b = ws1.cpu().numpy(), ws2.cpu().numpy()
    assert a[:4].view(np.uint32)[0] == 0 and b[:4].view(np.uint32)[0] == 0   # no device flags
    tpr = -(-V // (2048 // (2 if w.dtype == "bf16" else 4)))
    kb = w.k_per_row if getattr(w, "k_per_row", None) is not None else np.full(B, K)
    read = []
    for r in range(B):
        read += [r * (K + 1) + t for t in range(kb[r] + 1)]
        if w.temperature[r] > 0:
            read += [B * (K + 1) + r * K + t for t in range(kb[r])]
    for row in read:
        o = 256 + row * tpr * 8
        np.testing.assert_array_equal(a[o:o + tpr * 8], b[o:o + tpr * 8], err_msg=f"row {row}")


# ---------------------------------------------------------------- small shapes and edges

def _random_workload(rng, B, K, V, dtype, temps, neg_inf=False, ties=False):
    tg = rng.normal(0, 2.0, (B, K + 1, V))
    dr = tg[:, :K] + rng.normal(0, 0.7, (B, K, V))
    if ties:
        tg = np.round(tg)           # many equal logits: greedy ties
    if neg_inf:
        mask = rng.random((B, K + 1, V)) < 0.2
        mask[..., 0] = False        # keep one finite logit per row
        tg[mask] = -np.inf
        dmask = rng.random((B, K, V)) < 0.2
        dmask[..., 0] = False
        dr[dmask] = -np.inf
    w = synth.custom(tg, dr, np.zeros((B, K), np.int32), np.zeros((B, K + 1)),
                     np.asarray(temps, np.float32)[:B], dtype=dtype)
    # drafted tokens: from q for tempered rows (Gumbel-max on the stored values),
    # argmax of the draft for greedy rows, sometimes the target's argmax
    d64 = (w.draft.astype(np.uint32) << 16).view(np.float32).astype(np.float64) if dtype == "bf16" \
        else w.draft.astype(np.float64)
    t64 = (w.target.astype(np.uint32) << 16).view(np.float32).astype(np.float64) if dtype == "bf16" \
        else w.target.astype(np.float64)
    for b in range(B):
        for t in range(K):
            T = float(w.temperature[b])
            if T == 0 or rng.random() < 0.3:
                w.draft_tokens[b, t] = int(np.argmax(t64[b, t] if rng.random() < 0.7 else d64[b, t]))
            else:
                with np.errstate(divide="ignore"):
                    g = -np.log(-np.log(rng.random(V)))
                w.draft_tokens[b, t] = int(np.argmax(d64[b, t] / T + g))
    w.uniforms[:] = (rng.integers(0, 1 << 24, (B, K + 1)) * 2.0 ** -24).astype(np.float32)
    return w


CASES = [
    # (B, K, V, dtype, offset)
    (3, 1, 1, "f32", 0), (3, 2, 2, "bf16", 0), (5, 3, 7, "f32", 0), (4, 16, 33, "bf16", 0),
    (7, 4, 1000, "f32", 0), (6, 5, 4099, "bf16", 0), (5, 2, 8191, "f32", 0),
    (9, 3, 8192, "bf16", 0), (3, 6, 20000, "bf16", 1), (3, 4, 17001, "f32", 3),
    (2, 2, 65536, "bf16", 0), (2, 3, 70001, "f32", 0),
    # rows of many tiles: chunks of 4 tiles with a ragged last chunk and tile
    (32, 2, 140000, "bf16", 0), (33, 2, 140000, "bf16", 0),
    (4, 4, 128256, "bf16", 0), (9, 3, 100000, "bf16", 0), (10, 3, 100000, "bf16", 0),
    (1, 4, 32000, "bf16", 0), (16, 2, 32000, "bf16", 0), (3, 4, 9000, "f32", 5),
    # exactly one chunk per row, and one tile more
    (5, 3, 4096, "bf16", 0), (5, 3, 4097, "bf16", 0), (5, 3, 2048, "f32", 0),
    # the largest vocabularies accepted (1024 tiles per row) and the largest K
    (2, 2, 1 << 20, "bf16", 0), (2, 2, 1 << 19, "f32", 0), (2, 16, 128256, "bf16", 0),
]


@pytest.mark.parametrize("B,K,V,dtype,offset", CASES)
def test_small_shapes_match_oracle(B, K, V, dtype, offset):
    rng = np.random.default_rng(B * 1000 + K * 10 + V)
    temps = [0.0, 1.0, 0.3, 2.5, 0.7, 1.3, 0.0, 1.0, 0.9]
    total = None
    for variant in range(3):
        w = _random_workload(rng, B, K, V, dtype, np.resize(np.roll(temps, variant), B),
                             neg_inf=variant == 1, ties=variant == 2)
        g = run_gpu(w, offset_elems=offset)
        ref = run_oracle(w, workers=1)
        assert not check_structure(g["accepted"], g["out_tokens"], w.draft_tokens, w.V)
        rep = compare(ref, g["accepted"], g["out_tokens"], g["logp"], g["logq"], w.temperature)
        total = rep if total is None else total.merge(rep)
    _assert_parity(total, 0)


def test_error_rows_and_device_flags():
    import torch
    from speculative_decoding_verification_25_gb300 import _native as N
    from speculative_decoding_verification_25_gb300 import api
    rng = np.random.default_rng(0)
    B, K, V = 6, 3, 300
    w = _random_workload(rng, B, K, V, "f32", [1.0] * B)
    w.temperature[1] = -1.0
    w.temperature[2] = np.nan
    w.temperature[3] = 1e-39
    w.draft_tokens[4, 1] = V
    w.draft_tokens[5, 0] = -1
    d = device_tensors(w)
    ws = api.workspace_for(B, K, V, N.SV_F32, d["target"].device)
    res = api.spec_verify(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                          d["temperature"], want_logprobs=True, workspace=ws)
    flags = api.device_errors(ws)
    al = res.accepted_len.cpu().numpy()
    ot = res.out_tokens.cpu().numpy()
    assert al[0] >= 0
    assert (al[1:] == -1).all() and (ot[1:] == -1).all()
    assert flags == N.SV_DEV_BAD_TEMPERATURE | N.SV_DEV_BAD_TOKEN
    assert np.isnan(res.logp.cpu().numpy()[1:]).all()
    ref = run_oracle(w, workers=1)
    assert np.array_equal(ref.accepted_len, al) and np.array_equal(ref.out_tokens, ot)
    # a clean call on the same workspace clears the flags
    w2 = _random_workload(rng, B, K, V, "f32", [1.0] * B)
    d2 = device_tensors(w2)
    api.spec_verify(d2["target"], d2["draft"], d2["draft_tokens"], d2["uniforms"],
                    d2["temperature"], workspace=ws)
    assert api.device_errors(ws) == 0
    torch.cuda.synchronize()


def test_q_equal_p_accepts_every_draft():
    rng = np.random.default_rng(3)
    B, K, V = 16, 5, 3000
    tg = rng.normal(0, 2, (B, K + 1, V))
    w = synth.custom(tg, tg[:, :K], rng.integers(0, V, (B, K)),
                     rng.random((B, K + 1)) * 0.999, np.ones(B), dtype="bf16")
    g = run_gpu(w)
    assert (g["accepted"] == K).all()
    ref = run_oracle(w, workers=1)
    rep = compare(ref, g["accepted"], g["out_tokens"], g["logp"], g["logq"], w.temperature)
    _assert_parity(rep, 0)


def test_repeated_calls_are_deterministic_on_a_side_stream():
    import torch
    from speculative_decoding_verification_25_gb300 import api
    w = synth.make("llama3_stochastic", seed=5, rows=range(16))
    d = device_tensors(w)
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for _ in range(3):
            r = api.spec_verify(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                                d["temperature"], want_logprobs=True)
            outs.append([x.clone() for x in r])
    s.synchronize()
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert torch.equal(a, b)


# ---------------------------------------------------------------- statistics of the GPU path

def _shared_dists_workload(rng, B, logP, logQ):
    """B rows that all verify the same per-position distributions p_t, q_t
    (given as log-probabilities, used directly as logits at T = 1)."""
    K, V = logQ.shape
    Q = np.exp(logQ)
    tg = np.broadcast_to(logP, (B, K + 1, V))
    dr = np.broadcast_to(logQ, (B, K, V))
    tokens = np.stack([rng.choice(V, size=B, p=Q[t] / Q[t].sum()) for t in range(K)], axis=1)
    unif = (rng.integers(0, 1 << 24, (B, K + 1)) * 2.0 ** -24)
    return synth.custom(tg, dr, tokens, unif, np.ones(B), dtype="f32")


def test_gpu_emitted_tokens_follow_p_chi_square():
    scipy_stats = pytest.importorskip("scipy.stats")
    from oracle import oracle
    rng = np.random.default_rng(21)
    K, V, B = 3, 8, 1 << 18
    tg = rng.normal(0, 1.2, (K + 1, V))
    dr = tg[:K] + rng.normal(0, 1.2, (K, V))
    logP = np.stack([oracle.log_softmax(tg[t], 1.0) for t in range(K + 1)])
    logQ = np.stack([oracle.log_softmax(dr[t], 1.0) for t in range(K)])
    w = _shared_dists_workload(rng, B, logP.astype(np.float32), logQ.astype(np.float32))
    # the distributions the GPU actually sees are those of the stored float32 logits
    P = np.exp(np.stack([oracle.log_softmax(w.target[0, t].astype(np.float64), 1.0)
                         for t in range(K + 1)]))
    g = run_gpu(w, want_logprobs=False)
    n = g["accepted"]
    assert (n >= 0).all()
    for s in range(K + 1):
        sel = n >= s
        c = np.bincount(g["out_tokens"][sel, s], minlength=V)
        m = c.sum()
        stat, pval = scipy_stats.chisquare(c, m * P[s])
        assert pval > 1e-3, (s, pval)
        assert 0.5 * np.abs(c / m - P[s]).sum() < 0.01


def test_gpu_expected_tokens_alpha_08():
    rng = np.random.default_rng(8)
    K, B = 4, 1 << 18
    logP = np.log(np.tile([0.9, 0.1], (K + 1, 1)))
    logQ = np.log(np.tile([0.7, 0.3], (K, 1)))
    w = _shared_dists_workload(rng, B, logP, logQ)
    g = run_gpu(w, want_logprobs=False)
    tokens = g["accepted"] + 1
    E = 3.3616
    ps = np.array([0.8 ** j * 0.2 for j in range(K)] + [0.8 ** K])
    var = (ps * np.arange(1, K + 2) ** 2).sum() - E ** 2
    assert abs(tokens.mean() - E) < 4 * np.sqrt(var / B)
    # and the law of accepted_len is the truncated geometric one
    hist = np.bincount(g["accepted"], minlength=K + 1) / B
    assert np.abs(hist - ps).max() < 0.005
