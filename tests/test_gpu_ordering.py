"""Stream order around the launches that may start early (programmatic
dependent launch): when a kernel on the same stream writes the inputs just
before the call, every read of the call sees the written values.  The last
writer of each input here is an elementwise kernel, not a copy, so the
launch that follows it is a programmatic dependent of that kernel."""
import numpy as np
import pytest

from speculative_decoding_verification_25_gb300 import synth

from gpu_util import device_tensors

pytestmark = pytest.mark.gpu


def _overwrite_with_kernels(dst, src):
    # fill with junk, then add the real values: two kernels, the last one writes dst
    dst.fill_(7 if not dst.is_floating_point() else 3.0)
    dst.mul_(0).add_(src)


@pytest.mark.parametrize("name", ["llama3_stochastic", "llama3_ragged", "greedy_batch"])
def test_inputs_written_just_before_the_call_are_seen(name):
    import torch
    from speculative_decoding_verification_25_gb300 import api
    want_w = synth.make(name, seed=7, rows=range(16))
    junk_w = synth.make(name, seed=8, rows=range(16))
    want_d = device_tensors(want_w)
    bufs = device_tensors(junk_w)          # same shapes, other values
    torch.cuda.synchronize()

    want = api.spec_verify(want_d["target"], want_d["draft"], want_d["draft_tokens"],
                           want_d["uniforms"], want_d["temperature"],
                           k_per_row=want_d.get("k_per_row"), want_logprobs=True)
    B = want_w.B
    tok0 = torch.zeros(B, 32, dtype=torch.int32, device="cuda:0")
    L0 = torch.full((B,), 3, dtype=torch.int32, device="cuda:0")
    api.plug(want, tok0, L0)
    torch.cuda.synchronize()

    for step in range(3):   # repeated, so the previous call's kernels precede too
        for k, v in want_d.items():
            _overwrite_with_kernels(bufs[k], v)
        got = api.spec_verify(bufs["target"], bufs["draft"], bufs["draft_tokens"],
                              bufs["uniforms"], bufs["temperature"],
                              k_per_row=bufs.get("k_per_row"), want_logprobs=True)
        tok = torch.full((B, 32), 5, dtype=torch.int32, device="cuda:0")
        L = torch.full((B,), 9, dtype=torch.int32, device="cuda:0")
        tok.mul_(0)                        # the plug's inputs, also written by kernels
        L.mul_(0).add_(3)
        api.plug(got, tok, L)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got.accepted_len.cpu().numpy(), want.accepted_len.cpu().numpy())
        np.testing.assert_array_equal(got.out_tokens.cpu().numpy(), want.out_tokens.cpu().numpy())
        np.testing.assert_array_equal(got.logp.cpu().numpy().view(np.uint32),
                                      want.logp.cpu().numpy().view(np.uint32))
        np.testing.assert_array_equal(tok.cpu().numpy(), tok0.cpu().numpy())
        np.testing.assert_array_equal(L.cpu().numpy(), L0.cpu().numpy())


def test_two_streams_with_the_default_workspace_do_not_share_it():
    # the Python API caches one workspace per (device, stream): calls on
    # two streams may run at the same time and must not race on scratch
    import torch
    from speculative_decoding_verification_25_gb300 import api
    ws_ = [synth.make("llama3_stochastic", seed=s, rows=range(32)) for s in (11, 12)]
    d = [device_tensors(w) for w in ws_]
    want = []
    for di in d:
        r = api.spec_verify(di["target"], di["draft"], di["draft_tokens"], di["uniforms"],
                            di["temperature"], want_logprobs=True)
        torch.cuda.synchronize()
        want.append((r.accepted_len.cpu().numpy(), r.out_tokens.cpu().numpy(),
                     r.logp.cpu().numpy()))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for rnd in range(4):
        res = []
        for i, s in enumerate(streams):
            with torch.cuda.stream(s):
                di = d[i]
                res.append(api.spec_verify(di["target"], di["draft"], di["draft_tokens"],
                                           di["uniforms"], di["temperature"], want_logprobs=True))
        torch.cuda.synchronize()
        for r, (acc, out, lp) in zip(res, want):
            np.testing.assert_array_equal(r.accepted_len.cpu().numpy(), acc)
            np.testing.assert_array_equal(r.out_tokens.cpu().numpy(), out)
            np.testing.assert_array_equal(r.logp.cpu().numpy().view(np.uint32), lp.view(np.uint32))
