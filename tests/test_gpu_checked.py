"""The checked build (libspec_verify_checked.so, compiled with -DSV_CHECKED)
on small and odd shapes, through the C ABI: every global index the verify
kernel forms is tested against its buffer before the access, and a failed
test would set SV_DEV_OUT_OF_BOUNDS instead of faulting.  No call here may
raise that flag, and the outputs must still match the oracle."""
from __future__ import annotations

import numpy as np
import pytest

from speculative_decoding_verification_25_gb300 import synth

from _parity import check_structure, compare
from gpu_util import device_tensors, run_oracle
from test_gpu_parity import CASES, _random_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import torch
    from speculative_decoding_verification_25_gb300 import _native as N
    from speculative_decoding_verification_25_gb300 import build as b
    b.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return N.load_checked()


def _run_checked(lib, w, offset_elems=0):
    """One call of the checked library's spec_verify (spec_verify_ragged for
    a ragged workload); returns the outputs and the call's device flags."""
    import ctypes
    import torch
    from speculative_decoding_verification_25_gb300 import _native as N
    d = device_tensors(w, offset_elems=offset_elems)
    dt = N.SV_BF16 if w.dtype == "bf16" else N.SV_F32
    B, K, V = w.B, w.K, w.V
    nb = lib.spec_verify_workspace_bytes(B, K, V, dt)
    ws = torch.full((nb,), 0xAB, dtype=torch.uint8, device="cuda:0")   # garbage
    acc = torch.empty(B, dtype=torch.int32, device="cuda:0")
    out = torch.empty(B, K + 1, dtype=torch.int32, device="cuda:0")
    lp = torch.empty(B, K, dtype=torch.float32, device="cuda:0")
    lq = torch.empty(B, K, dtype=torch.float32, device="cuda:0")
    sh = torch.cuda.current_stream().cuda_stream
    common = (d["draft_tokens"].data_ptr(), d["uniforms"].data_ptr(), d["temperature"].data_ptr())
    tail = (acc.data_ptr(), out.data_ptr(), lp.data_ptr(), lq.data_ptr(), ws.data_ptr(), nb, sh)
    if "k_per_row" in d:
        st = lib.spec_verify_ragged(d["target"].data_ptr(), d["draft"].data_ptr(), dt, *common,
                                    d["k_per_row"].data_ptr(), B, K, V, *tail)
    else:
        st = lib.spec_verify(d["target"].data_ptr(), d["draft"].data_ptr(), dt, *common, B, K, V,
                             *tail)
    assert st == N.SV_OK, N.status_string(st)
    flags = ctypes.c_uint32(0)
    assert lib.spec_verify_device_errors(ws.data_ptr(), sh, ctypes.byref(flags)) == N.SV_OK
    return dict(accepted=acc.cpu().numpy(), out_tokens=out.cpu().numpy(), logp=lp.cpu().numpy(),
                logq=lq.cpu().numpy(), flags=int(flags.value))


def _check(w, g, max_mismatch=0):
    from speculative_decoding_verification_25_gb300 import _native as N
    assert not g["flags"] & N.SV_DEV_OUT_OF_BOUNDS, hex(g["flags"])
    assert not check_structure(g["accepted"], g["out_tokens"], w.draft_tokens, w.V)
    rep = compare(run_oracle(w, workers=1), g["accepted"], g["out_tokens"], g["logp"], g["logq"],
                  w.temperature)
    assert not rep.failures, rep.failures[:5]
    assert rep.mismatched_rows <= max_mismatch, rep


@pytest.mark.parametrize("B,K,V,dtype,offset", CASES)
def test_checked_build_small_shapes(lib, B, K, V, dtype, offset):
    rng = np.random.default_rng(B * 1000 + K * 10 + V + 7)
    temps = [0.0, 1.0, 0.3, 2.5, 0.7, 1.3, 0.0, 1.0, 0.9]
    for variant in range(2):
        w = _random_workload(rng, B, K, V, dtype, np.resize(np.roll(temps, variant), B),
                             neg_inf=variant == 1)
        _check(w, _run_checked(lib, w, offset))


@pytest.mark.parametrize("name,rows", [("tiny_stochastic", None), ("tiny_greedy", None),
                                       ("greedy_batch", range(9)), ("llama3_stochastic", range(20)),
                                       ("llama3_ragged", range(33)), ("long_draft_mixed_t", range(11))])
def test_checked_build_workload_rows(lib, name, rows):
    w = synth.make(name, seed=3, rows=rows)
    _check(w, _run_checked(lib, w))


def test_checked_build_error_rows(lib):
    from speculative_decoding_verification_25_gb300 import _native as N
    rng = np.random.default_rng(5)
    w = _random_workload(rng, 5, 3, 700, "f32", [1.0, -1.0, 1.0, 0.0, 1.0])
    w.draft_tokens[2, 0] = 700
    g = _run_checked(lib, w)
    assert g["flags"] == N.SV_DEV_BAD_TEMPERATURE | N.SV_DEV_BAD_TOKEN
    assert list(g["accepted"][[1, 2]]) == [-1, -1]
    ref = run_oracle(w, workers=1)
    np.testing.assert_array_equal(ref.accepted_len, g["accepted"])
    np.testing.assert_array_equal(ref.out_tokens, g["out_tokens"])
