"""Adaptive verification (spec_verify_ragged): the CUDA path against the
oracle's spec_verify_ragged on the same seeded inputs."""
import dataclasses

import numpy as np
import pytest

from speculative_decoding_verification_25_gb300 import synth

from _parity import check_structure, compare
from gpu_util import device_tensors, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def _assert_parity(rep):
    assert not rep.failures, rep.failures[:5]
    assert rep.mismatched_rows == 0, rep


def test_llama3_ragged_full_size():
    w = synth.make("llama3_ragged", seed=0, workers=synth.default_workers())
    g = run_gpu(w)
    ref = run_oracle(w)
    assert not check_structure(g["accepted"], g["out_tokens"], w.draft_tokens, w.V)
    assert (g["accepted"] <= w.k_per_row).all()
    _assert_parity(compare(ref, g["accepted"], g["out_tokens"], g["logp"], g["logq"], w.temperature))


def _random(rng, B, K, V, dtype, kb):
    tg = rng.normal(0, 2.0, (B, K + 1, V))
    dr = tg[:, :K] + rng.normal(0, 0.7, (B, K, V))
    temps = rng.choice([0.0, 0.6, 1.0, 1.4], B).astype(np.float32)
    tok = np.empty((B, K), np.int32)
    for b in range(B):
        for t in range(K):
            z = dr[b, t] / max(float(temps[b]), 1.0)
            pr = np.exp(z - z.max())
            tok[b, t] = rng.choice(V, p=pr / pr.sum())
    unif = rng.random((B, K + 1)).astype(np.float32)
    w = synth.custom(tg, dr, tok, unif, temps, dtype=dtype)
    return dataclasses.replace(w, k_per_row=np.asarray(kb, np.int32))


@pytest.mark.parametrize("B,K,V,dtype", [(24, 4, 3000, "f32"), (20, 6, 4099, "bf16"),
                                         (9, 16, 257, "f32"), (17, 3, 1, "bf16")])
def test_small_shapes_every_row_length(B, K, V, dtype):
    rng = np.random.default_rng(B * 7 + K)
    w = _random(rng, B, K, V, dtype, [b % (K + 1) for b in range(B)])
    g = run_gpu(w)
    ref = run_oracle(w, workers=1)
    assert (g["accepted"] <= w.k_per_row).all()
    _assert_parity(compare(ref, g["accepted"], g["out_tokens"], g["logp"], g["logq"], w.temperature))


def test_full_length_everywhere_equals_spec_verify_bit_for_bit():
    w = synth.make("llama3_stochastic", seed=3, rows=range(16))
    a = run_gpu(w)
    b = run_gpu(dataclasses.replace(w, k_per_row=np.full(w.B, w.K, np.int32)))
    for k in ("accepted", "out_tokens"):
        np.testing.assert_array_equal(a[k], b[k])
    np.testing.assert_array_equal(a["logp"].view(np.uint32), b["logp"].view(np.uint32))


def test_rows_past_the_prefix_are_never_read():
    # NaN in every target row past K_b and every draft row at or past K_b:
    # a read would poison the row statistics (and flag the row)
    rng = np.random.default_rng(5)
    B, K, V = 12, 5, 2048
    kb = np.array([b % (K + 1) for b in range(B)], np.int32)
    w = _random(rng, B, K, V, "f32", kb)
    tg, dr = w.target.copy(), w.draft.copy()
    for b in range(B):
        tg[b, kb[b] + 1:] = np.nan
        dr[b, kb[b]:] = np.nan
    clean = run_oracle(w, workers=1)
    w2 = dataclasses.replace(w, target=tg, draft=dr)
    g = run_gpu(w2)
    assert (g["accepted"] >= 0).all()
    _assert_parity(compare(clean, g["accepted"], g["out_tokens"], g["logp"], g["logq"], w.temperature))


def test_bad_lengths_are_error_rows_with_a_flag():
    import torch
    from speculative_decoding_verification_25_gb300 import api, _native as N
    rng = np.random.default_rng(6)
    w = _random(rng, 4, 3, 500, "f32", [-1, 4, 3, 0])
    d = device_tensors(w)
    ws = api.workspace_for(w.B, w.K, w.V, N.SV_F32, d["target"].device)
    r = api.spec_verify(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                        d["temperature"], k_per_row=d["k_per_row"], workspace=ws)
    torch.cuda.synchronize()
    acc = r.accepted_len.cpu().numpy()
    assert list(acc[:2]) == [-1, -1]
    assert (r.out_tokens.cpu().numpy()[:2] == -1).all()
    assert acc[2] >= 0 and acc[3] == 0
    assert api.device_errors(ws) & N.SV_DEV_BAD_K


@pytest.mark.parametrize("B,dtype", [(2048, "f32"), (2049, "bf16")])
def test_large_ragged_batches(B, dtype):
    # thousands of short rows: many batch rows per chunk window, most
    # chunks one tile, rows of every length
    rng = np.random.default_rng(B)
    K, V = 3, 600
    w = _random(rng, B, K, V, dtype, rng.integers(0, K + 1, B))
    g = run_gpu(w)
    ref = run_oracle(w)
    assert (g["accepted"] <= w.k_per_row).all()
    _assert_parity(compare(ref, g["accepted"], g["out_tokens"], g["logp"], g["logq"], w.temperature))


def test_greedy_rows_without_lengths_skip_their_draft_rows():
    # the chunks of a greedy row's draft rows are skipped by the warps they
    # fall to
    rng = np.random.default_rng(11)
    w = _random(rng, 40, 5, 5000, "bf16", np.full(40, 5))
    w = dataclasses.replace(w, k_per_row=None)
    assert (w.temperature == 0).any() and (w.temperature > 0).any()
    g = run_gpu(w)
    ref = run_oracle(w)
    _assert_parity(compare(ref, g["accepted"], g["out_tokens"], g["logp"], g["logq"], w.temperature))
