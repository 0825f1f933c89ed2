"""ctypes binding of libspec_verify.so: the C ABI of include/spec_verify.h,
same names, argument marshalling only.  Every step of the verify path runs
in the library's CUDA kernels; if the library is missing this module raises
instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libspec_verify.so")
# the same library compiled with index checks (tests only)
LIB_CHECKED_PATH = os.path.join(PKG, "libspec_verify_checked.so")

SV_F32 = 0
SV_BF16 = 1

SV_OK = 0
SV_ERR_NULL = 1
SV_ERR_SHAPE = 2
SV_ERR_DTYPE = 3
SV_ERR_ALIGN = 4
SV_ERR_WORKSPACE = 5
SV_ERR_CUDA = 6
SV_ERR_TOO_LARGE = 7

SV_DEV_BAD_TEMPERATURE = 1
SV_DEV_BAD_TOKEN = 2
SV_DEV_NONFINITE = 4
SV_DEV_BAD_K = 8
SV_DEV_PLUG_CLIPPED = 16
SV_DEV_BAD_LENGTH = 32
SV_DEV_BAD_TREE = 64
SV_DEV_OUT_OF_BOUNDS = 256

SV_MAX_K = 16
SV_MAX_TREE_NODES = 128
SV_STATIC_SCRATCH_BYTES = 8 << 20

# every function of include/spec_verify.h: (restype, argtypes)
_P = ctypes.c_void_p
_I = ctypes.c_int
_SIG = {
    "spec_verify_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "spec_verify_max_vocab": (_I, [_I]),
    "spec_verify": (_I, [_P, _P, _I, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P,
                         ctypes.c_size_t, _P]),
    "spec_verify_device_errors": (_I, [_P, _P, ctypes.POINTER(ctypes.c_uint32)]),
    "spec_verify_static": (_I, [_P, _P, _I, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "spec_verify_tree_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "spec_verify_tree": (_I, [_P, _I, _P, _P, _I, _I, _I, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "spec_verify_plug": (_I, [_P, _P, _I, _I, _P, _P, _I, _P, _P, _P]),
    "spec_verify_ragged": (_I, [_P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P,
                                ctypes.c_size_t, _P]),
    "spec_verify_and_plug": (_I, [_P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P,
                                  _I, _P, _P, ctypes.c_size_t, _P]),
    "spec_verify_status_string": (ctypes.c_char_p, [_I]),
    "spec_verify_row_stats": (_I, [_P, _P, _I, _P, _P, _I, _I, _I, _P, ctypes.c_size_t, _P]),
    "spec_verify_static_device_errors": (_I, [_P, ctypes.POINTER(ctypes.c_uint32)]),
}

_lib = None
_lib_checked = None


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, what: str = "spec_verify"):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_string(status)})")


def load() -> ctypes.CDLL:
    """Load the in-tree library (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
        _lib = _open(LIB_PATH)
    return _lib


def _open(path: str) -> ctypes.CDLL:
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIG.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load_checked() -> ctypes.CDLL:
    """The checked build (every kernel index tested against its buffer; a
    failure sets SV_DEV_OUT_OF_BOUNDS), with the same C entry points."""
    global _lib_checked
    if _lib_checked is None:
        if not os.path.exists(LIB_CHECKED_PATH):
            raise ImportError(f"{LIB_CHECKED_PATH} is not built")
        _lib_checked = _open(LIB_CHECKED_PATH)
    return _lib_checked


def spec_verify_workspace_bytes(B: int, K: int, V: int, dtype: int) -> int:
    return int(load().spec_verify_workspace_bytes(B, K, V, dtype))


def spec_verify_max_vocab(dtype: int) -> int:
    return int(load().spec_verify_max_vocab(dtype))


def status_string(status: int) -> str:
    return load().spec_verify_status_string(status).decode()


spec_verify_status_string = status_string


def spec_verify_raw(target_ptr, draft_ptr, dtype, tokens_ptr, uniforms_ptr, temperature_ptr,
                    B, K, V, accepted_ptr, out_tokens_ptr, logp_ptr, logq_ptr,
                    workspace_ptr, workspace_bytes, stream_handle) -> int:
    """The C entry point with plain integer addresses; returns the status."""
    return int(load().spec_verify(target_ptr, draft_ptr, dtype, tokens_ptr, uniforms_ptr,
                                  temperature_ptr, B, K, V, accepted_ptr, out_tokens_ptr,
                                  logp_ptr, logq_ptr, workspace_ptr, workspace_bytes,
                                  stream_handle))


def spec_verify_row_stats_raw(target_ptr, draft_ptr, dtype, temperature_ptr, k_per_row_ptr, B, K,
                              V, workspace_ptr, workspace_bytes, stream_handle) -> int:
    """The streaming launch of spec_verify alone (k_per_row_ptr 0: all K)."""
    return int(load().spec_verify_row_stats(target_ptr, draft_ptr, dtype, temperature_ptr,
                                            k_per_row_ptr or None, B, K, V, workspace_ptr,
                                            workspace_bytes, stream_handle))


def spec_verify_ragged_raw(target_ptr, draft_ptr, dtype, tokens_ptr, uniforms_ptr,
                           temperature_ptr, k_per_row_ptr, B, K, V, accepted_ptr, out_tokens_ptr,
                           logp_ptr, logq_ptr, workspace_ptr, workspace_bytes, stream_handle) -> int:
    """spec_verify with a per-row number of verified drafts (k_per_row)."""
    return int(load().spec_verify_ragged(target_ptr, draft_ptr, dtype, tokens_ptr, uniforms_ptr,
                                         temperature_ptr, k_per_row_ptr, B, K, V, accepted_ptr,
                                         out_tokens_ptr, logp_ptr, logq_ptr, workspace_ptr,
                                         workspace_bytes, stream_handle))


def spec_verify_and_plug_raw(target_ptr, draft_ptr, dtype, tokens_ptr, uniforms_ptr,
                             temperature_ptr, k_per_row_ptr, B, K, V, accepted_ptr,
                             out_tokens_ptr, logp_ptr, logq_ptr, seq_tokens_ptr, seq_len_ptr,
                             max_len, last_token_ptr, workspace_ptr, workspace_bytes,
                             stream_handle) -> int:
    """spec_verify (ragged if k_per_row is given) with the plug step fused in."""
    return int(load().spec_verify_and_plug(
        target_ptr, draft_ptr, dtype, tokens_ptr, uniforms_ptr, temperature_ptr, k_per_row_ptr,
        B, K, V, accepted_ptr, out_tokens_ptr, logp_ptr, logq_ptr, seq_tokens_ptr, seq_len_ptr,
        max_len, last_token_ptr, workspace_ptr, workspace_bytes, stream_handle))


def spec_verify_tree_workspace_bytes(B: int, N: int, V: int, dtype: int) -> int:
    return int(load().spec_verify_tree_workspace_bytes(B, N, V, dtype))


def spec_verify_tree_raw(target_ptr, dtype, node_tokens_ptr, parents_ptr, B, N, V, accepted_ptr,
                         out_tokens_ptr, accepted_nodes_ptr, workspace_ptr, workspace_bytes,
                         stream_handle) -> int:
    """Greedy verification of one draft tree per row."""
    return int(load().spec_verify_tree(target_ptr, dtype, node_tokens_ptr, parents_ptr, B, N, V,
                                       accepted_ptr, out_tokens_ptr, accepted_nodes_ptr,
                                       workspace_ptr, workspace_bytes, stream_handle))


def spec_verify_plug_raw(accepted_ptr, out_tokens_ptr, B, K, tokens_ptr, seq_len_ptr, max_len,
                         last_token_ptr, flags_ptr, stream_handle) -> int:
    """Append emitted tokens to the per-row sequences on the device."""
    return int(load().spec_verify_plug(accepted_ptr, out_tokens_ptr, B, K, tokens_ptr, seq_len_ptr,
                                       max_len, last_token_ptr, flags_ptr, stream_handle))


def spec_verify_static_raw(target_ptr, draft_ptr, dtype, tokens_ptr, uniforms_ptr,
                           temperature_ptr, B, K, V, accepted_ptr, out_tokens_ptr, logp_ptr,
                           logq_ptr, stream_handle) -> int:
    """spec_verify on the library's static scratch (no workspace argument)."""
    return int(load().spec_verify_static(target_ptr, draft_ptr, dtype, tokens_ptr, uniforms_ptr,
                                         temperature_ptr, B, K, V, accepted_ptr, out_tokens_ptr,
                                         logp_ptr, logq_ptr, stream_handle))


def spec_verify_device_errors(workspace_ptr, stream_handle) -> int:
    flags = ctypes.c_uint32(0)
    st = int(load().spec_verify_device_errors(workspace_ptr, stream_handle, ctypes.byref(flags)))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_device_errors")
    return int(flags.value)
