"""spec_verify_static (the entry point that allocates nothing and works in
the library's own static device scratch) against spec_verify on the same
inputs, through the C ABI.  Kept in its own file, collected last, so that
it runs both on a fresh process and after every other GPU test."""
import numpy as np
import pytest

from speculative_decoding_verification_25_gb300 import synth

from gpu_util import device_tensors

pytestmark = pytest.mark.gpu


def _outputs(B, K, device):
    import torch
    return (torch.empty(B, dtype=torch.int32, device=device),
            torch.empty(B, K + 1, dtype=torch.int32, device=device),
            torch.empty(B, K, dtype=torch.float32, device=device),
            torch.empty(B, K, dtype=torch.float32, device=device))


def _host(outs):
    return [t.cpu().numpy() for t in outs]


@pytest.mark.parametrize("name,rows", [("llama3_stochastic", range(64)), ("tiny_stochastic", None),
                                       ("greedy_batch", range(8))])
def test_static_scratch_matches_spec_verify_twice_in_a_row(name, rows):
    import torch
    from speculative_decoding_verification_25_gb300 import _native as N
    w = synth.make(name, seed=5, rows=rows)
    d = device_tensors(w)
    dt = N.SV_BF16 if w.dtype == "bf16" else N.SV_F32
    B, K, V = w.B, w.K, w.V
    assert N.spec_verify_workspace_bytes(B, K, V, dt) <= N.SV_STATIC_SCRATCH_BYTES
    stream = torch.cuda.current_stream().cuda_stream
    ptrs = [d[k].data_ptr() for k in ("target", "draft")]
    ins = [d[k].data_ptr() for k in ("draft_tokens", "uniforms", "temperature")]

    # the existing entry point on a caller workspace
    nbytes = N.spec_verify_workspace_bytes(B, K, V, dt)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda:0")
    ref = _outputs(B, K, "cuda:0")
    st = N.spec_verify_raw(ptrs[0], ptrs[1], dt, *ins, B, K, V, *[t.data_ptr() for t in ref],
                           ws.data_ptr(), nbytes, stream)
    assert st == N.SV_OK, N.status_string(st)

    # two static calls in a row on the same stream, into fresh outputs
    got = []
    for _ in range(2):
        outs = _outputs(B, K, "cuda:0")
        st = N.spec_verify_static_raw(ptrs[0], ptrs[1], dt, *ins, B, K, V,
                                      *[t.data_ptr() for t in outs], stream)
        assert st == N.SV_OK, N.status_string(st)
        got.append(outs)
    torch.cuda.synchronize()

    acc_r, tok_r, lp_r, lq_r = _host(ref)
    assert (acc_r >= 0).all()
    for outs in got:
        acc, tok, lp, lq = _host(outs)
        np.testing.assert_array_equal(acc, acc_r)
        np.testing.assert_array_equal(tok, tok_r)
        sampled = w.temperature > 0
        np.testing.assert_allclose(lp[sampled], lp_r[sampled], rtol=0, atol=1e-5)
        np.testing.assert_allclose(lq[sampled], lq_r[sampled], rtol=0, atol=1e-5)
        assert np.isnan(lp[~sampled]).all() and np.isnan(lq[~sampled]).all()

    # and the calls allocate nothing: the device's free memory is the same
    # before and after a run of them (outputs allocated beforehand)
    outs = _outputs(B, K, "cuda:0")
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(20):
        st = N.spec_verify_static_raw(ptrs[0], ptrs[1], dt, *ins, B, K, V,
                                      *[t.data_ptr() for t in outs], stream)
        assert st == N.SV_OK, N.status_string(st)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    np.testing.assert_array_equal(_host(outs)[1], tok_r)


def test_static_scratch_rejects_a_shape_beyond_its_size():
    from speculative_decoding_verification_25_gb300 import _native as N
    B = 1
    while N.spec_verify_workspace_bytes(B, 4, 128256, N.SV_BF16) <= N.SV_STATIC_SCRATCH_BYTES:
        B += 1
    # the pointers are never used: the size check comes before any launch
    st = N.spec_verify_static_raw(0x10000, 0x10000, N.SV_BF16, 0x10000, 0x10000, 0x10000, B, 4,
                                  128256, 0x10000, 0x10000, None, None, None)
    assert st == N.SV_ERR_TOO_LARGE


def test_static_device_flags_are_readable():
    """spec_verify_static_device_errors returns the flags of the last static
    call: a bad temperature and a bad token raise theirs, a clean call
    clears them."""
    import ctypes
    import torch
    from speculative_decoding_verification_25_gb300 import _native as N
    lib = N.load()
    w = synth.make("llama3_stochastic", seed=6, rows=range(6))
    stream = torch.cuda.current_stream().cuda_stream
    B, K, V = w.B, w.K, w.V

    def run(temps, tokens):
        d = device_tensors(w)
        d["temperature"].copy_(torch.tensor(temps, dtype=torch.float32))
        d["draft_tokens"].copy_(torch.from_numpy(tokens))
        outs = _outputs(B, K, "cuda:0")
        st = N.spec_verify_static_raw(d["target"].data_ptr(), d["draft"].data_ptr(), N.SV_BF16,
                                      d["draft_tokens"].data_ptr(), d["uniforms"].data_ptr(),
                                      d["temperature"].data_ptr(), B, K, V,
                                      *[t.data_ptr() for t in outs], stream)
        assert st == N.SV_OK, N.status_string(st)
        flags = ctypes.c_uint32(0xFFFFFFFF)
        assert lib.spec_verify_static_device_errors(stream, ctypes.byref(flags)) == N.SV_OK
        return int(flags.value), outs[0].cpu().numpy()

    bad_tokens = w.draft_tokens.copy()
    bad_tokens[3, 1] = V
    flags, acc = run([1.0, -1.0, 1.0, 1.0, 0.0, 1.0], bad_tokens)
    assert flags == N.SV_DEV_BAD_TEMPERATURE | N.SV_DEV_BAD_TOKEN
    assert acc[1] == -1 and acc[3] == -1 and (np.delete(acc, [1, 3]) >= 0).all()
    flags, acc = run(list(w.temperature), w.draft_tokens)
    assert flags == 0 and (acc >= 0).all()
    assert lib.spec_verify_static_device_errors(stream, None) == N.SV_ERR_NULL
