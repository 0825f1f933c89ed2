"""Test-side helpers: move a synthetic workload to the GPU, run the CUDA path
through the C ABI, and run the oracle on chosen rows (in a spawn pool)."""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np


def device_tensors(w, device="cuda:0", offset_elems=0):
    """Workload -> CUDA tensors.  ``offset_elems`` > 0 places the logits that
    many elements past a 16-byte boundary (exercises the scalar path)."""
    import torch
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def logits(a):
        host = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if w.dtype == "bf16" else a)
        if w.dtype == "bf16":
            host = host.view(torch.bfloat16)
        if offset_elems:
            buf = torch.empty(host.numel() + offset_elems, dtype=dt, device=device)
            t = buf[offset_elems:].view(host.shape)
            t.copy_(host)
            return t
        return host.to(device)

    d = dict(target=logits(w.target), draft=logits(w.draft),
             draft_tokens=torch.from_numpy(w.draft_tokens).to(device),
             uniforms=torch.from_numpy(w.uniforms).to(device),
             temperature=torch.from_numpy(w.temperature).to(device))
    if getattr(w, "k_per_row", None) is not None:
        d["k_per_row"] = torch.from_numpy(np.ascontiguousarray(w.k_per_row, np.int32)).to(device)
    return d


def run_gpu(w, device="cuda:0", offset_elems=0, want_logprobs=True):
    import torch
    from speculative_decoding_verification_25_gb300 import api
    d = device_tensors(w, device, offset_elems)
    res = api.spec_verify(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                          d["temperature"], k_per_row=d.get("k_per_row"),
                          want_logprobs=want_logprobs)
    torch.cuda.synchronize()
    out = dict(accepted=res.accepted_len.cpu().numpy(), out_tokens=res.out_tokens.cpu().numpy(),
               logp=res.logp.cpu().numpy() if want_logprobs else None,
               logq=res.logq.cpu().numpy() if want_logprobs else None)
    del d, res
    return out


def _oracle_job(args):
    target, draft, tokens, unif, temp, dtype, kpr = args
    from oracle import oracle
    if kpr is not None:
        return oracle.spec_verify_ragged(target, draft, tokens, unif, temp, kpr, dtype=dtype)
    return oracle.spec_verify(target, draft, tokens, unif, temp, dtype=dtype)


def run_oracle(w, rows=None, workers=None):
    """Oracle on batch rows ``rows`` of workload ``w`` (indices into w)."""
    from oracle import oracle
    rows = np.arange(w.B) if rows is None else np.asarray(rows)
    workers = workers or max(1, min(16, os.cpu_count() or 1))
    chunks = [c for c in np.array_split(rows, min(workers, len(rows))) if len(c)]
    kpr = getattr(w, "k_per_row", None)
    jobs = [(w.target[c], w.draft[c], w.draft_tokens[c], w.uniforms[c], w.temperature[c], w.dtype,
             None if kpr is None else kpr[c]) for c in chunks]
    if len(jobs) == 1:
        parts = [_oracle_job(jobs[0])]
    else:
        with mp.get_context("spawn").Pool(len(jobs)) as pool:
            parts = pool.map(_oracle_job, jobs)
    cat = lambda f: np.concatenate([getattr(p, f) for p in parts])
    return oracle.BatchResult(cat("accepted_len"), cat("out_tokens"), cat("logp"), cat("logq"),
                              cat("ratio_margin"), cat("cdf_margin"),
                              sum((p.mode for p in parts), []))


def _workload_oracle_job(args):
    name, seed, rows = args
    from oracle import oracle
    from speculative_decoding_verification_25_gb300 import synth
    w = synth.make(name, seed=seed, rows=rows)
    kpr = getattr(w, "k_per_row", None)
    if kpr is not None:
        return oracle.spec_verify_ragged(w.target, w.draft, w.draft_tokens, w.uniforms,
                                         w.temperature, kpr, dtype=w.dtype)
    return oracle.spec_verify(w.target, w.draft, w.draft_tokens, w.uniforms, w.temperature,
                              dtype=w.dtype)


def run_oracle_workload(name, seed, B, workers=None):
    """The oracle on every row of a named synthetic workload.  Each worker
    rebuilds its own rows from the seed (the generator draws every row from
    streams of its own), so no logits cross process boundaries."""
    from oracle import oracle
    workers = workers or max(1, min(16, os.cpu_count() or 1))
    chunks = [c for c in np.array_split(np.arange(B), min(workers * 4, B)) if len(c)]
    with mp.get_context("spawn").Pool(min(workers, len(chunks))) as pool:
        parts = pool.map(_workload_oracle_job, [(name, seed, c) for c in chunks])
    cat = lambda f: np.concatenate([getattr(p, f) for p in parts])
    return oracle.BatchResult(cat("accepted_len"), cat("out_tokens"), cat("logp"), cat("logq"),
                              cat("ratio_margin"), cat("cdf_margin"),
                              sum((p.mode for p in parts), []))
