"""Greedy tree verification on the GPU against the oracle (bit-exact)."""
import numpy as np
import pytest

from speculative_decoding_verification_25_gb300 import synth

pytestmark = pytest.mark.gpu


def _gpu_tree(target_raw, dtype, tokens, parents, offset_elems=0):
    import torch
    from speculative_decoding_verification_25_gb300 import api
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    host = torch.from_numpy(np.ascontiguousarray(target_raw).view(np.int16) if dtype == "bf16"
                            else np.ascontiguousarray(target_raw))
    if dtype == "bf16":
        host = host.view(torch.bfloat16)
    if offset_elems:
        buf = torch.empty(host.numel() + offset_elems, dtype=dt, device="cuda:0")
        tg = buf[offset_elems:].view(host.shape)
        tg.copy_(host)
    else:
        tg = host.to("cuda:0")
    r = api.verify_tree(tg, torch.from_numpy(np.ascontiguousarray(tokens, np.int32)).cuda(),
                        torch.from_numpy(np.ascontiguousarray(parents, np.int32)).cuda(),
                        want_nodes=True)
    torch.cuda.synchronize()
    return r.accepted_len.cpu().numpy(), r.out_tokens.cpu().numpy(), r.accepted_nodes.cpu().numpy()


def _check(ref, got):
    np.testing.assert_array_equal(got[0], ref.accepted_len)
    np.testing.assert_array_equal(got[1], ref.out_tokens)
    np.testing.assert_array_equal(got[2], ref.accepted_nodes)


def test_llama3_tree_full_size_bit_exact():
    from oracle import oracle
    w = synth.make("llama3_tree", seed=0, workers=synth.default_workers())
    got = _gpu_tree(w.target, w.dtype, w.draft_tokens, w.parents)
    ref = oracle.verify_tree_greedy(w.target, w.draft_tokens, w.parents, dtype=w.dtype)
    assert (ref.accepted_len >= 2).sum() > 5          # the workload does accept paths
    _check(ref, got)


@pytest.mark.parametrize("B,N,V,dtype,offset", [(8, 1, 7, "f32", 0), (12, 30, 4099, "bf16", 0),
                                               (5, 128, 513, "f32", 1), (9, 64, 2048, "bf16", 3)])
def test_random_trees(B, N, V, dtype, offset):
    from oracle import oracle
    rng = np.random.default_rng(N + V)
    tg = rng.normal(0, 2, (B, N + 1, V))
    if dtype == "bf16":
        tg[:, :, :3] = 9.0                            # ties at the top: lowest index wins
    raw = synth.custom(tg, np.zeros((B, N, V)), np.zeros((B, N), np.int32),
                       np.zeros((B, N + 1)), np.zeros(B), dtype=dtype).target
    stored = oracle.decode_logits(raw, dtype)
    am = stored.argmax(axis=2)
    par = np.array([[int(rng.integers(-1, i)) for i in range(N)] for _ in range(B)], np.int32)
    tok = np.empty((B, N), np.int32)
    for b in range(B):
        for i in range(N):
            slot = 0 if par[b, i] < 0 else par[b, i] + 1
            tok[b, i] = am[b, slot] if rng.random() < 0.7 else rng.integers(0, V)
    got = _gpu_tree(raw, dtype, tok, par, offset)
    ref = oracle.verify_tree_greedy(raw, tok, par, dtype=dtype)
    _check(ref, got)


def test_chain_tree_matches_spec_verify_greedy():
    import torch
    from speculative_decoding_verification_25_gb300 import api
    w = synth.make("greedy_batch", seed=1, rows=range(16))
    par = np.tile(np.arange(w.K, dtype=np.int32) - 1, (w.B, 1))
    acc, out, _ = _gpu_tree(w.target, w.dtype, w.draft_tokens, par)
    from gpu_util import run_gpu
    g = run_gpu(w)
    np.testing.assert_array_equal(acc, g["accepted"])
    np.testing.assert_array_equal(out, g["out_tokens"])


def test_malformed_trees_are_flagged():
    import torch
    from speculative_decoding_verification_25_gb300 import api, _native as N
    V, Nn = 300, 4
    tg = torch.randn(3, Nn + 1, V, device="cuda:0")
    tok = torch.tensor([[0, 1, 2, 3], [0, 1, 2, 3], [0, 1, 2, 999]], dtype=torch.int32).cuda()
    par = torch.tensor([[-1, 0, 1, 2], [-1, 1, 0, 0], [-1, 0, 0, 0]], dtype=torch.int32).cuda()
    ws = torch.empty(N.spec_verify_tree_workspace_bytes(3, Nn, V, N.SV_F32), dtype=torch.uint8,
                     device="cuda:0")
    r = api.verify_tree(tg, tok, par, workspace=ws)
    torch.cuda.synchronize()
    acc = r.accepted_len.cpu().numpy()
    assert acc[0] >= 0 and acc[1] == -1 and acc[2] == -1
    assert (r.out_tokens.cpu().numpy()[1:] == -1).all()
    assert api.device_errors(ws) & N.SV_DEV_BAD_TREE
