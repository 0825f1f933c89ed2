"""Torch-facing wrapper of the C ABI.  PyTorch supplies device memory and
streams; the verify step itself runs in the library's kernels.

    accepted_len, out_tokens = spec_verify(target, draft, draft_tokens,
                                           uniforms, temperature)

``target`` [B, K+1, V] and ``draft`` [B, K, V] are CUDA tensors of
torch.bfloat16 or torch.float32; ``draft_tokens`` [B, K] int32;
``uniforms`` [B, K+1] float32; ``temperature`` [B] float32 (0 = greedy).
"""
from __future__ import annotations

from typing import NamedTuple, Optional

import torch

from . import _native as N
from . import _native as _N

_DTYPES = {torch.bfloat16: N.SV_BF16, torch.float32: N.SV_F32}
_workspaces: dict = {}


class VerifyResult(NamedTuple):
    accepted_len: torch.Tensor           # [B] int32, -1 = error row
    out_tokens: torch.Tensor             # [B, K+1] int32, -1 padded
    logp: Optional[torch.Tensor] = None  # [B, K] float32 log p_t(x_t)
    logq: Optional[torch.Tensor] = None  # [B, K] float32 log q_t(x_t)


def _check(t: torch.Tensor, name: str, dtype=None, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def workspace_for(B: int, K: int, V: int, dtype: int, device: torch.device,
                  stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """A cached device workspace large enough for this shape, one per
    (device, stream): calls on one stream run in order and may share it,
    calls on different streams may overlap and must not."""
    need = N.spec_verify_workspace_bytes(B, K, V, dtype)
    if need == 0:
        raise ValueError(f"invalid shape B={B} K={K} V={V}")
    index = device.index if device.index is not None else torch.cuda.current_device()
    st = stream if stream is not None else torch.cuda.current_stream(index)
    key = (index, st.cuda_stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < need:
        with torch.cuda.stream(st):   # allocated for use on this stream
            ws = torch.empty(max(need, 1 << 20), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def spec_verify(target: torch.Tensor, draft: torch.Tensor, draft_tokens: torch.Tensor,
                uniforms: torch.Tensor, temperature: torch.Tensor, *,
                k_per_row: Optional[torch.Tensor] = None,
                want_logprobs: bool = False, out: Optional[VerifyResult] = None,
                workspace: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> VerifyResult:
    """Verify a batch on the current (or given) CUDA stream; no host sync.

    ``k_per_row`` ([B] int32, optional): row b verifies only its first
    k_per_row[b] drafted tokens (adaptive verification, spec_verify_ragged).
    """
    if target.dim() != 3:
        raise ValueError("target must be [B, K+1, V]")
    B, K1, V = target.shape
    K = K1 - 1
    dev = target.device
    if target.dtype not in _DTYPES:
        raise TypeError(f"target dtype {target.dtype} is not bfloat16 or float32")
    dt = _DTYPES[target.dtype]
    _check(target, "target", device=dev)
    _check(draft, "draft", dtype=target.dtype, shape=(B, K, V), device=dev)
    _check(draft_tokens, "draft_tokens", dtype=torch.int32, shape=(B, K), device=dev)
    _check(uniforms, "uniforms", dtype=torch.float32, shape=(B, K + 1), device=dev)
    _check(temperature, "temperature", dtype=torch.float32, shape=(B,), device=dev)
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    if out is None:
        with torch.cuda.stream(st):   # outputs belong to the stream that writes them
            out = VerifyResult(
                torch.empty(B, dtype=torch.int32, device=dev),
                torch.empty(B, K + 1, dtype=torch.int32, device=dev),
                torch.empty(B, K, dtype=torch.float32, device=dev) if want_logprobs else None,
                torch.empty(B, K, dtype=torch.float32, device=dev) if want_logprobs else None)
    if workspace is None:
        workspace = workspace_for(B, K, V, dt, dev, st)
    lp = out.logp.data_ptr() if out.logp is not None else None
    lq = out.logq.data_ptr() if out.logq is not None else None
    ws_bytes = workspace.numel() * workspace.element_size()
    if k_per_row is None:
        status = N.spec_verify_raw(
            target.data_ptr(), draft.data_ptr(), dt, draft_tokens.data_ptr(), uniforms.data_ptr(),
            temperature.data_ptr(), B, K, V, out.accepted_len.data_ptr(),
            out.out_tokens.data_ptr(), lp, lq, workspace.data_ptr(), ws_bytes, st.cuda_stream)
    else:
        _check(k_per_row, "k_per_row", dtype=torch.int32, shape=(B,), device=dev)
        status = N.spec_verify_ragged_raw(
            target.data_ptr(), draft.data_ptr(), dt, draft_tokens.data_ptr(), uniforms.data_ptr(),
            temperature.data_ptr(), k_per_row.data_ptr(), B, K, V, out.accepted_len.data_ptr(),
            out.out_tokens.data_ptr(), lp, lq, workspace.data_ptr(), ws_bytes, st.cuda_stream)
    if status != N.SV_OK:
        raise N.SpecVerifyError(status)
    return out


def device_errors(workspace: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> int:
    """SV_DEV_* flags of the last call on ``workspace`` (synchronises the stream)."""
    st = stream if stream is not None else torch.cuda.current_stream(workspace.device)
    return N.spec_verify_device_errors(workspace.data_ptr(), st.cuda_stream)


def plug(result: VerifyResult, tokens: torch.Tensor, seq_len: torch.Tensor, *,
         last_token: Optional[torch.Tensor] = None, flags: Optional[torch.Tensor] = None,
         stream: Optional[torch.cuda.Stream] = None) -> None:
    """Append each row's emitted tokens to ``tokens`` [B, max_len] (int32) at
    ``seq_len`` [B] (int32, advanced in place) on the device; no host sync.
    ``last_token`` [B] int32 receives each row's last emitted token;
    ``flags`` (one int32) collects SV_DEV_PLUG_CLIPPED / SV_DEV_BAD_LENGTH."""
    B, K1 = result.out_tokens.shape
    dev = result.out_tokens.device
    if tokens.dim() != 2 or tokens.shape[0] != B:
        raise ValueError("tokens must be [B, max_len]")
    _check(tokens, "tokens", dtype=torch.int32, device=dev)
    _check(seq_len, "seq_len", dtype=torch.int32, shape=(B,), device=dev)
    if last_token is not None:
        _check(last_token, "last_token", dtype=torch.int32, shape=(B,), device=dev)
    if flags is not None:
        _check(flags, "flags", dtype=torch.int32, shape=(1,), device=dev)
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    status = N.spec_verify_plug_raw(
        result.accepted_len.data_ptr(), result.out_tokens.data_ptr(), B, K1 - 1,
        tokens.data_ptr(), seq_len.data_ptr(), tokens.shape[1],
        last_token.data_ptr() if last_token is not None else None,
        flags.data_ptr() if flags is not None else None, st.cuda_stream)
    if status != N.SV_OK:
        raise N.SpecVerifyError(status, "spec_verify_plug")


def spec_verify_and_plug(target: torch.Tensor, draft: torch.Tensor, draft_tokens: torch.Tensor,
                         uniforms: torch.Tensor, temperature: torch.Tensor, tokens: torch.Tensor,
                         seq_len: torch.Tensor, *, k_per_row: Optional[torch.Tensor] = None,
                         last_token: Optional[torch.Tensor] = None,
                         want_logprobs: bool = False, out: Optional[VerifyResult] = None,
                         workspace: Optional[torch.Tensor] = None,
                         stream: Optional[torch.cuda.Stream] = None) -> VerifyResult:
    """spec_verify followed by plug, with the plug step fused into the
    verify call's second launch (same results as the two calls).  Plug flags
    go to the workspace word: read them with ``device_errors(workspace)``."""
    if target.dim() != 3:
        raise ValueError("target must be [B, K+1, V]")
    B, K1, V = target.shape
    K = K1 - 1
    dev = target.device
    if target.dtype not in _DTYPES:
        raise TypeError(f"target dtype {target.dtype} is not bfloat16 or float32")
    dt = _DTYPES[target.dtype]
    _check(target, "target", device=dev)
    _check(draft, "draft", dtype=target.dtype, shape=(B, K, V), device=dev)
    _check(draft_tokens, "draft_tokens", dtype=torch.int32, shape=(B, K), device=dev)
    _check(uniforms, "uniforms", dtype=torch.float32, shape=(B, K + 1), device=dev)
    _check(temperature, "temperature", dtype=torch.float32, shape=(B,), device=dev)
    if tokens.dim() != 2 or tokens.shape[0] != B:
        raise ValueError("tokens must be [B, max_len]")
    _check(tokens, "tokens", dtype=torch.int32, device=dev)
    _check(seq_len, "seq_len", dtype=torch.int32, shape=(B,), device=dev)
    if last_token is not None:
        _check(last_token, "last_token", dtype=torch.int32, shape=(B,), device=dev)
    if k_per_row is not None:
        _check(k_per_row, "k_per_row", dtype=torch.int32, shape=(B,), device=dev)
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    if out is None:
        with torch.cuda.stream(st):   # outputs belong to the stream that writes them
            out = VerifyResult(
                torch.empty(B, dtype=torch.int32, device=dev),
                torch.empty(B, K + 1, dtype=torch.int32, device=dev),
                torch.empty(B, K, dtype=torch.float32, device=dev) if want_logprobs else None,
                torch.empty(B, K, dtype=torch.float32, device=dev) if want_logprobs else None)
    if workspace is None:
        workspace = workspace_for(B, K, V, dt, dev, st)
    status = N.spec_verify_and_plug_raw(
        target.data_ptr(), draft.data_ptr(), dt, draft_tokens.data_ptr(), uniforms.data_ptr(),
        temperature.data_ptr(), k_per_row.data_ptr() if k_per_row is not None else None, B, K, V,
        out.accepted_len.data_ptr(), out.out_tokens.data_ptr(),
        out.logp.data_ptr() if out.logp is not None else None,
        out.logq.data_ptr() if out.logq is not None else None,
        tokens.data_ptr(), seq_len.data_ptr(), tokens.shape[1],
        last_token.data_ptr() if last_token is not None else None,
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), st.cuda_stream)
    if status != N.SV_OK:
        raise N.SpecVerifyError(status, "spec_verify_and_plug")
    return out


class TreeResult(NamedTuple):
    accepted_len: torch.Tensor                  # [B] int32: depth of the accepted path, -1 = error row
    out_tokens: torch.Tensor                    # [B, N+1] int32: path tokens, bonus, -1 padded
    accepted_nodes: Optional[torch.Tensor] = None   # [B, N] int32: path node indices, -1 padded


def verify_tree(target: torch.Tensor, node_tokens: torch.Tensor, parents: torch.Tensor, *,
                want_nodes: bool = False, workspace: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> TreeResult:
    """Greedy verification of one draft tree per row (spec_verify_tree):
    ``target`` [B, N+1, V] (slot 0 after the context, slot i+1 after node i),
    ``node_tokens`` and ``parents`` [B, N] int32 (parents[b, i] in [-1, i))."""
    if target.dim() != 3:
        raise ValueError("target must be [B, N+1, V]")
    B, N1, V = target.shape
    N = N1 - 1
    dev = target.device
    if target.dtype not in _DTYPES:
        raise TypeError(f"target dtype {target.dtype} is not bfloat16 or float32")
    dt = _DTYPES[target.dtype]
    _check(target, "target", device=dev)
    _check(node_tokens, "node_tokens", dtype=torch.int32, shape=(B, N), device=dev)
    _check(parents, "parents", dtype=torch.int32, shape=(B, N), device=dev)
    need = _N.spec_verify_tree_workspace_bytes(B, N, V, dt)
    if need == 0:
        raise ValueError(f"invalid tree shape B={B} N={N} V={V}")
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.stream(st):   # blocks the allocator may reuse only after st's work
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        res = TreeResult(torch.empty(B, dtype=torch.int32, device=dev),
                         torch.empty(B, N + 1, dtype=torch.int32, device=dev),
                         torch.empty(B, N, dtype=torch.int32, device=dev) if want_nodes else None)
    status = _N.spec_verify_tree_raw(
        target.data_ptr(), dt, node_tokens.data_ptr(), parents.data_ptr(), B, N, V,
        res.accepted_len.data_ptr(), res.out_tokens.data_ptr(),
        res.accepted_nodes.data_ptr() if res.accepted_nodes is not None else None,
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), st.cuda_stream)
    if status != _N.SV_OK:
        raise _N.SpecVerifyError(status, "spec_verify_tree")
    return res
