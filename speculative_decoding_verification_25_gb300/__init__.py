"""Batched speculative-decoding verify-and-accept on GB300 (sm_103a).

The C ABI lives in include/spec_verify.h and libspec_verify.so (built
in-tree by ``build.build()``); ``api.spec_verify`` is the torch-facing call.
"""
from . import _native  # noqa: F401


def spec_verify(*args, **kwargs):
    """See :func:`speculative_decoding_verification_25_gb300.api.spec_verify`."""
    from .api import spec_verify as _sv
    return _sv(*args, **kwargs)
