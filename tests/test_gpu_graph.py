"""The verify step and the plug step captured in one CUDA graph: replays on
new inputs give exactly what eager calls give.  The first eager call sets up
the device (SM count, kernel attributes); after it, neither entry point
makes a call that stream capture forbids."""
import numpy as np
import pytest

from speculative_decoding_verification_25_gb300 import synth

from gpu_util import device_tensors

pytestmark = pytest.mark.gpu

MAX_LEN, START = 48, 7


def _eager(d, api):
    import torch
    B, K = d["draft_tokens"].shape
    res = api.spec_verify(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                          d["temperature"], k_per_row=d.get("k_per_row"))
    tokens = torch.full((B, MAX_LEN), -1, dtype=torch.int32, device="cuda:0")
    seq_len = torch.full((B,), START, dtype=torch.int32, device="cuda:0")
    api.plug(res, tokens, seq_len)
    torch.cuda.synchronize()
    return (res.accepted_len.cpu().numpy(), res.out_tokens.cpu().numpy(), tokens.cpu().numpy(),
            seq_len.cpu().numpy())


@pytest.mark.parametrize("name", ["llama3_stochastic", "llama3_ragged"])
def test_verify_and_plug_replay_in_a_cuda_graph(name):
    import torch
    from speculative_decoding_verification_25_gb300 import api
    from speculative_decoding_verification_25_gb300 import _native as N
    ws = [synth.make(name, seed=s, rows=range(16)) for s in (0, 1)]
    inputs = [device_tensors(w) for w in ws]
    want = [_eager(d, api) for d in inputs]

    # static buffers the graph reads and writes
    w = ws[0]
    B, K, V = w.B, w.K, w.V
    static = {k: v.clone() for k, v in inputs[0].items()}
    nb = N.spec_verify_workspace_bytes(B, K, V, N.SV_BF16)
    workspace = torch.zeros(nb, dtype=torch.uint8, device="cuda:0")
    out = api.VerifyResult(torch.empty(B, dtype=torch.int32, device="cuda:0"),
                           torch.empty(B, K + 1, dtype=torch.int32, device="cuda:0"))
    tokens = torch.full((B, MAX_LEN), -1, dtype=torch.int32, device="cuda:0")
    seq_len = torch.full((B,), START, dtype=torch.int32, device="cuda:0")

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        api.spec_verify(static["target"], static["draft"], static["draft_tokens"],
                        static["uniforms"], static["temperature"],
                        k_per_row=static.get("k_per_row"), out=out, workspace=workspace)
        api.plug(out, tokens, seq_len)

    for i in (1, 0, 1):   # new inputs each replay, copied into the static buffers
        for k, v in inputs[i].items():
            static[k].copy_(v)
        tokens.fill_(-1)
        seq_len.fill_(START)
        g.replay()
        torch.cuda.synchronize()
        got = (out.accepted_len.cpu().numpy(), out.out_tokens.cpu().numpy(),
               tokens.cpu().numpy(), seq_len.cpu().numpy())
        for a, b in zip(got, want[i]):
            np.testing.assert_array_equal(a, b)
    assert (want[0][3] == START + want[0][0] + 1).all()
