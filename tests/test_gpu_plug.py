"""The plug step on the GPU against the oracle's plug (bit-exact)."""
import numpy as np
import pytest

from speculative_decoding_verification_25_gb300 import synth

from _parity import compare
from gpu_util import device_tensors, run_oracle

pytestmark = pytest.mark.gpu


def _states(rng, B, K, max_len):
    acc = rng.integers(-1, K + 1, B).astype(np.int32)
    out = np.full((B, K + 1), -1, np.int32)
    for b in range(B):
        if acc[b] >= 0:
            out[b, :acc[b] + 1] = rng.integers(0, 50000, acc[b] + 1)
    tok = rng.integers(0, 50000, (B, max_len)).astype(np.int32)
    L = rng.integers(0, max_len + 1, B).astype(np.int32)
    L[:3] = [max_len - 1, max_len, 0]
    L[3:5] = [-1, max_len + 1]      # outside the buffer: left unchanged, flagged
    acc[5:7] = [K + 1, 31]          # not a length the verify step writes: unchanged, flagged
    return acc, out, tok, L


def test_plug_matches_the_oracle_bit_for_bit():
    import torch
    from speculative_decoding_verification_25_gb300 import _native as N
    from oracle import oracle
    rng = np.random.default_rng(0)
    B, K, max_len = 300, 5, 64
    acc, out, tok, L = _states(rng, B, K, max_len)
    dev = "cuda:0"
    t_acc, t_out = torch.from_numpy(acc).to(dev), torch.from_numpy(out).to(dev)
    t_tok, t_L = torch.from_numpy(tok).to(dev), torch.from_numpy(L).to(dev)
    t_last = torch.full((B,), -7, dtype=torch.int32, device=dev)
    t_flags = torch.zeros(1, dtype=torch.int32, device=dev)
    st = N.spec_verify_plug_raw(t_acc.data_ptr(), t_out.data_ptr(), B, K, t_tok.data_ptr(),
                                t_L.data_ptr(), max_len, t_last.data_ptr(), t_flags.data_ptr(),
                                torch.cuda.current_stream().cuda_stream)
    assert st == N.SV_OK
    torch.cuda.synchronize()
    ref = oracle.plug(acc, out, tok, L, last_token=np.full(B, -7, np.int32))
    np.testing.assert_array_equal(t_tok.cpu().numpy(), ref.tokens)
    np.testing.assert_array_equal(t_L.cpu().numpy(), ref.seq_len)
    np.testing.assert_array_equal(t_last.cpu().numpy(), ref.last_token)
    flags = int(t_flags.item())
    assert bool(flags & N.SV_DEV_PLUG_CLIPPED) == bool(ref.clipped.any())
    assert flags & N.SV_DEV_BAD_LENGTH


def test_verify_then_plug_on_the_device():
    import torch
    from speculative_decoding_verification_25_gb300 import api
    from oracle import oracle
    w = synth.make("llama3_stochastic", seed=4, rows=range(24))
    d = device_tensors(w)
    rng = np.random.default_rng(1)
    max_len = 40
    tok = rng.integers(0, w.V, (w.B, max_len)).astype(np.int32)
    L = rng.integers(0, max_len - w.K, w.B).astype(np.int32)
    t_tok = torch.from_numpy(tok).to("cuda:0")
    t_L = torch.from_numpy(L).to("cuda:0")
    last = torch.empty(w.B, dtype=torch.int32, device="cuda:0")
    r = api.spec_verify(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], d["temperature"],
                        want_logprobs=True)
    api.plug(r, t_tok, t_L, last_token=last)          # same stream, no host read in between
    torch.cuda.synchronize()
    ref = run_oracle(w, workers=1)
    rep = compare(ref, r.accepted_len.cpu().numpy(), r.out_tokens.cpu().numpy(),
                  r.logp.cpu().numpy(), r.logq.cpu().numpy(), w.temperature)
    assert not rep.failures and rep.mismatched_rows == 0
    want = oracle.plug(ref.accepted_len, ref.out_tokens, tok, L)
    np.testing.assert_array_equal(t_tok.cpu().numpy(), want.tokens)
    np.testing.assert_array_equal(t_L.cpu().numpy(), want.seq_len)
    np.testing.assert_array_equal(last.cpu().numpy(), want.last_token)


@pytest.mark.parametrize("name,rows", [("llama3_stochastic", range(24)), ("greedy_batch", range(32)),
                                       ("llama3_ragged", range(24)),
                                       ("long_draft_mixed_t", range(0, 240, 10))])
def test_fused_plug_equals_verify_then_plug(name, rows):
    import torch
    from speculative_decoding_verification_25_gb300 import api, _native as N
    w = synth.make(name, seed=2, rows=rows)
    d = device_tensors(w)
    if name == "llama3_stochastic":
        d["temperature"][3] = -1.0                  # an error row: never plugged
    B, K = w.B, w.K
    rng = np.random.default_rng(3)
    max_len = 3 * (K + 1)
    tok0 = rng.integers(0, 1000, (B, max_len)).astype(np.int32)
    L0 = rng.integers(0, max_len - K, B).astype(np.int32)
    L0[:3] = [max_len - 1, max_len, -1]             # clipped, full, outside the buffer
    kpr = d.get("k_per_row")

    ref = api.spec_verify(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                          d["temperature"], k_per_row=kpr)
    t_ref, L_ref = torch.from_numpy(tok0).cuda(), torch.from_numpy(L0).cuda()
    last_ref = torch.full((B,), -9, dtype=torch.int32, device="cuda:0")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    api.plug(ref, t_ref, L_ref, last_token=last_ref, flags=flags)

    ws = torch.zeros(N.spec_verify_workspace_bytes(B, K, w.V, N.SV_BF16 if w.dtype == "bf16"
                                                   else N.SV_F32), dtype=torch.uint8,
                     device="cuda:0")
    t_f, L_f = torch.from_numpy(tok0).cuda(), torch.from_numpy(L0).cuda()
    last_f = torch.full((B,), -9, dtype=torch.int32, device="cuda:0")
    res = api.spec_verify_and_plug(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                                   d["temperature"], t_f, L_f, k_per_row=kpr, last_token=last_f,
                                   workspace=ws)
    dev_flags = api.device_errors(ws)
    torch.cuda.synchronize()
    for a, b in ((res.accepted_len, ref.accepted_len), (res.out_tokens, ref.out_tokens),
                 (t_f, t_ref), (L_f, L_ref), (last_f, last_ref)):
        np.testing.assert_array_equal(a.cpu().numpy(), b.cpu().numpy())
    ref_flags = int(flags.item())
    mask = N.SV_DEV_PLUG_CLIPPED | N.SV_DEV_BAD_LENGTH
    assert dev_flags & mask == ref_flags & mask
    assert ref_flags & N.SV_DEV_BAD_LENGTH and ref_flags & N.SV_DEV_PLUG_CLIPPED


@pytest.mark.parametrize("max_len", [1, 40])
def test_fused_plug_at_the_largest_k(max_len):
    # K = 16: up to 17 emitted tokens per row, one per lane of the plugging warp
    import torch
    from speculative_decoding_verification_25_gb300 import api
    rng = np.random.default_rng(16 + max_len)
    B, K, V = 9, 16, 257
    tg = rng.normal(0, 2.0, (B, K + 1, V))
    dr = tg[:, :K] + rng.normal(0, 0.05, (B, K, V))   # close drafts: long accepted runs
    temps = np.array([0.0, 1.0, 0.7, 1.0, 0.0, 1.3, 1.0, 0.9, 1.0], np.float32)
    tok = np.array([[int(np.argmax(dr[b, t])) for t in range(K)] for b in range(B)], np.int32)
    unif = rng.random((B, K + 1)).astype(np.float32)
    w = synth.custom(tg, dr, tok, unif, temps, dtype="f32")
    d = device_tensors(w)
    L0 = np.array([0, 3, max_len, 0, 1, 0, 2, 0, 0], np.int32).clip(0, max_len)
    ref = api.spec_verify(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                          d["temperature"])
    t_ref = torch.full((B, max_len), -3, dtype=torch.int32, device="cuda:0")
    L_ref = torch.from_numpy(L0).cuda()
    api.plug(ref, t_ref, L_ref)
    t_f = torch.full((B, max_len), -3, dtype=torch.int32, device="cuda:0")
    L_f = torch.from_numpy(L0).cuda()
    res = api.spec_verify_and_plug(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                                   d["temperature"], t_f, L_f)
    torch.cuda.synchronize()
    assert (ref.accepted_len.cpu().numpy() >= 8).any()   # some rows emit many tokens
    for a, b in ((res.accepted_len, ref.accepted_len), (res.out_tokens, ref.out_tokens),
                 (t_f, t_ref), (L_f, L_ref)):
        np.testing.assert_array_equal(a.cpu().numpy(), b.cpu().numpy())
