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
