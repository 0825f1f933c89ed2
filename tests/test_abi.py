"""The C ABI on the host: the library loads without a GPU, exports every
function include/spec_verify.h declares, and rejects bad arguments with a
status before anything is launched (no call here reaches the GPU)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def N():
    from speculative_decoding_verification_25_gb300 import build as b
    b.build()
    from speculative_decoding_verification_25_gb300 import _native
    _native.load()
    return _native


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M):
            if not m.group(0).lstrip().startswith(("#", "if", "return")):
                names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for required in ("spec_verify", "spec_verify_workspace_bytes", "spec_verify_status_string",
                     "spec_verify_device_errors", "spec_verify_max_vocab"):
        assert required in names


def test_every_declared_symbol_is_exported(N):
    lib = ctypes.CDLL(N.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert set(_declared_functions()) <= set(N._SIG)


def _layout_bytes(B, K, V, elt):
    """The workspace layout: a 256-byte header, then 256-byte aligned
    regions -- one 8-byte partial per 2 KB tile of every target and draft
    row, a 4-byte draw ticket per batch row, and a 32-byte record per tile
    of every batch row's sampled row."""
    al = lambda x: (x + 255) // 256 * 256
    rows = B * (2 * K + 1)
    tpr = -(-V // (2048 // elt))
    off = 256
    for size in (rows * tpr * 8, B * 4, B * tpr * 32):
        off = al(off + size)
    return off


def test_workspace_bytes_arithmetic(N):
    for B, K, V in ((64, 4, 128256), (1, 4, 1000), (512, 10, 262144), (3, 16, 33), (256, 8, 152064)):
        assert N.spec_verify_workspace_bytes(B, K, V, N.SV_BF16) == _layout_bytes(B, K, V, 2)
        assert N.spec_verify_workspace_bytes(B, K, V, N.SV_F32) == _layout_bytes(B, K, V, 4)
    assert N.spec_verify_workspace_bytes(0, 4, 1000, N.SV_F32) == _layout_bytes(0, 4, 1000, 4)
    for bad in ((-1, 4, 10, 0), (1, 0, 10, 0), (1, 17, 10, 0), (1, 4, 0, 0), (1, 4, 10, 2),
                (1, 4, N.spec_verify_max_vocab(0) + 1, 0)):
        assert N.spec_verify_workspace_bytes(*bad) == 0


def test_max_vocab_covers_the_workloads(N):
    assert N.spec_verify_max_vocab(N.SV_BF16) >= 262144
    assert N.spec_verify_max_vocab(N.SV_F32) >= 262144
    assert N.spec_verify_max_vocab(7) == 0


def test_status_strings(N):
    for s in range(8):
        assert N.status_string(s) != "unknown status"
    assert N.status_string(99) == "unknown status"


FAKE = 0x10000   # never dereferenced: every call below fails validation first


def _call(N, **kw):
    args = dict(target=FAKE, draft=FAKE, dtype=N.SV_BF16, tokens=FAKE, uniforms=FAKE,
                temperature=FAKE, B=2, K=4, V=1024, accepted=FAKE, out=FAKE, logp=None,
                logq=None, ws=FAKE, ws_bytes=1 << 30, stream=None)
    args.update(kw)
    return N.spec_verify_raw(args["target"], args["draft"], args["dtype"], args["tokens"],
                             args["uniforms"], args["temperature"], args["B"], args["K"],
                             args["V"], args["accepted"], args["out"], args["logp"],
                             args["logq"], args["ws"], args["ws_bytes"], args["stream"])


def test_validation_errors_launch_nothing(N):
    assert _call(N, dtype=5) == N.SV_ERR_DTYPE
    assert _call(N, B=-1) == N.SV_ERR_SHAPE
    assert _call(N, K=0) == N.SV_ERR_SHAPE
    assert _call(N, K=17) == N.SV_ERR_SHAPE
    assert _call(N, V=0) == N.SV_ERR_SHAPE
    assert _call(N, V=N.spec_verify_max_vocab(N.SV_BF16) + 1) == N.SV_ERR_SHAPE
    for field in ("target", "draft", "tokens", "uniforms", "temperature", "accepted", "out", "ws"):
        assert _call(N, **{field: None}) == N.SV_ERR_NULL, field
    assert _call(N, target=FAKE + 1) == N.SV_ERR_ALIGN          # bf16 needs 2-byte alignment
    assert _call(N, dtype=N.SV_F32, draft=FAKE + 2) == N.SV_ERR_ALIGN
    assert _call(N, tokens=FAKE + 2) == N.SV_ERR_ALIGN
    assert _call(N, logp=FAKE + 1) == N.SV_ERR_ALIGN
    assert _call(N, ws=FAKE + 8) == N.SV_ERR_ALIGN
    need = N.spec_verify_workspace_bytes(2, 4, 1024, N.SV_BF16)
    assert _call(N, ws_bytes=need - 1) == N.SV_ERR_WORKSPACE


def test_empty_batch_is_a_no_op(N):
    assert _call(N, B=0, target=None, draft=None, tokens=None, uniforms=None, temperature=None,
                 accepted=None, out=None, ws=None, ws_bytes=0) == N.SV_OK


def test_static_entry_point_rejects_before_touching_the_device(N):
    """spec_verify_static: argument and size checks come before any CUDA call."""
    def call(dtype=N.SV_BF16, B=2, K=4, V=1024):
        return N.spec_verify_static_raw(FAKE, FAKE, dtype, FAKE, FAKE, FAKE, B, K, V, FAKE, FAKE,
                                        None, None, None)
    assert call(dtype=5) == N.SV_ERR_DTYPE
    assert call(K=0) == N.SV_ERR_SHAPE
    assert call(B=-3) == N.SV_ERR_SHAPE
    assert call(B=0) == N.SV_OK
    # the largest batch at the Llama-3 vocabulary that fits the static scratch, and one more
    fits = [B for B in range(1, 4000)
            if N.spec_verify_workspace_bytes(B, 4, 128256, N.SV_BF16) <= N.SV_STATIC_SCRATCH_BYTES]
    assert fits and fits == list(range(1, fits[-1] + 1)) and fits[-1] >= 64
    assert call(B=fits[-1] + 1, V=128256) == N.SV_ERR_TOO_LARGE
    assert call(B=512, K=10, V=262144) == N.SV_ERR_TOO_LARGE
    assert "static" in N.status_string(N.SV_ERR_TOO_LARGE)


def test_device_errors_rejects_null(N):
    flags = ctypes.c_uint32(0)
    assert N.load().spec_verify_device_errors(None, None, ctypes.byref(flags)) == N.SV_ERR_NULL
    assert N.load().spec_verify_device_errors(FAKE, None, None) == N.SV_ERR_NULL


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from speculative_decoding_verification_25_gb300 import _native
    monkeypatch.setattr(_native, "_lib", None)
    monkeypatch.setattr(_native, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(ImportError):
        _native.load()


def test_ragged_entry_point_checks_its_length_array(N):
    def call(kpr, B=2):
        return N.spec_verify_ragged_raw(FAKE, FAKE, N.SV_BF16, FAKE, FAKE, FAKE, kpr, B, 4, 1024,
                                        FAKE, FAKE, None, None, FAKE, 1 << 30, None)
    assert call(None) == N.SV_ERR_NULL
    assert call(FAKE + 2) == N.SV_ERR_ALIGN
    assert call(None, B=0) == N.SV_OK
    assert N.spec_verify_ragged_raw(FAKE, FAKE, 9, FAKE, FAKE, FAKE, FAKE, 2, 4, 1024, FAKE, FAKE,
                                    None, None, FAKE, 1 << 30, None) == N.SV_ERR_DTYPE


def test_fused_plug_entry_point_checks_arguments(N):
    def call(**kw):
        a = dict(t=FAKE, d=FAKE, dt=N.SV_BF16, tok=FAKE, u=FAKE, T=FAKE, kpr=None, B=2, K=4, V=1024,
                 acc=FAKE, out=FAKE, seq=FAKE, L=FAKE, max_len=16, last=None, ws=FAKE, wsb=1 << 30)
        a.update(kw)
        return N.spec_verify_and_plug_raw(a["t"], a["d"], a["dt"], a["tok"], a["u"], a["T"],
                                          a["kpr"], a["B"], a["K"], a["V"], a["acc"], a["out"],
                                          None, None, a["seq"], a["L"], a["max_len"], a["last"],
                                          a["ws"], a["wsb"], None)
    assert call(B=0, seq=None, L=None) == N.SV_OK
    assert call(max_len=0) == N.SV_ERR_SHAPE
    assert call(seq=None) == N.SV_ERR_NULL
    assert call(L=None) == N.SV_ERR_NULL
    assert call(L=FAKE + 2) == N.SV_ERR_ALIGN
    assert call(last=FAKE + 1) == N.SV_ERR_ALIGN
    assert call(kpr=FAKE + 2) == N.SV_ERR_ALIGN
    assert call(dt=7) == N.SV_ERR_DTYPE
    assert call(wsb=16) == N.SV_ERR_WORKSPACE


def test_plug_entry_point_checks_arguments(N):
    def call(B=2, K=4, max_len=16, acc=FAKE, out=FAKE, tok=FAKE, L=FAKE, last=None, flags=None):
        return N.spec_verify_plug_raw(acc, out, B, K, tok, L, max_len, last, flags, None)
    assert call(B=0, acc=None, out=None, tok=None, L=None) == N.SV_OK
    assert call(B=-1) == N.SV_ERR_SHAPE
    assert call(K=0) == N.SV_ERR_SHAPE
    assert call(max_len=0) == N.SV_ERR_SHAPE
    for field in ("acc", "out", "tok", "L"):
        assert call(**{field: None}) == N.SV_ERR_NULL, field
    assert call(tok=FAKE + 2) == N.SV_ERR_ALIGN
    assert call(flags=FAKE + 1) == N.SV_ERR_ALIGN


def test_tree_entry_points_check_arguments(N):
    B, Nn, V = 64, 21, 128256
    tiles = -(-V // 1024)
    assert N.spec_verify_tree_workspace_bytes(B, Nn, V, N.SV_BF16) == 256 + B * (Nn + 1) * tiles * 8
    assert N.spec_verify_tree_workspace_bytes(B, 0, V, N.SV_BF16) == 0
    assert N.spec_verify_tree_workspace_bytes(B, N.SV_MAX_TREE_NODES + 1, V, N.SV_BF16) == 0

    def call(**kw):
        a = dict(t=FAKE, dt=N.SV_BF16, tok=FAKE, par=FAKE, B=2, n=4, V=1024, acc=FAKE, out=FAKE,
                 nodes=None, ws=FAKE, wsb=1 << 30)
        a.update(kw)
        return N.spec_verify_tree_raw(a["t"], a["dt"], a["tok"], a["par"], a["B"], a["n"], a["V"],
                                      a["acc"], a["out"], a["nodes"], a["ws"], a["wsb"], None)
    assert call(dt=7) == N.SV_ERR_DTYPE
    assert call(n=0) == N.SV_ERR_SHAPE
    assert call(B=0, t=None, tok=None, par=None, acc=None, out=None, ws=None) == N.SV_OK
    for f in ("t", "tok", "par", "acc", "out", "ws"):
        assert call(**{f: None}) == N.SV_ERR_NULL, f
    assert call(t=FAKE + 1) == N.SV_ERR_ALIGN
    assert call(nodes=FAKE + 2) == N.SV_ERR_ALIGN
    assert call(wsb=16) == N.SV_ERR_WORKSPACE
