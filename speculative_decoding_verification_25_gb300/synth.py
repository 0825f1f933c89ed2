"""Seeded synthetic workloads for the batched verify-and-accept step.

This module only *makes inputs*.  It holds none of the verification
arithmetic (no softmax, no acceptance test, no residual, no inverse CDF):
both the CPU oracle and the CUDA path consume what it produces, and neither
imports anything else from the other.

What the pages fix about the inputs (lesson "Decodificação Especulativa e
EAGLE", section "O Conceito / A Configuração com Dois Modelos"): the target
model gives logits at K+1 positions, the draft model at K positions, and the
K drafted tokens are sampled from the draft distribution q.  The five shapes
and value distributions below are the workloads this library is measured on;
the pages name no dataset, so every value here is synthetic.

Recipe (all randomness from numpy PCG64, one independent stream per
(workload, batch row, purpose, position), derived with
``SeedSequence(seed, spawn_key=...)`` so any subset of rows can be rebuilt
without generating the rest):

* logits are drawn in float64, then rounded once to the storage type
  (float32 by IEEE round-to-nearest-even; bf16 by rounding that float32 to
  the upper 16 bits, nearest-even).  Those stored values *are* the input for
  both sides.
* the draft row is built from the float64 target row before rounding.
* drafted tokens are sampled from the stored draft row at the row's
  temperature with the Gumbel-max construction
  ``argmax(d / T + G)``, ``G = -log(-log U)``, which is exact sampling from
  ``softmax(d / T)`` and shares nothing with the verify rule; a T = 0 row
  takes ``argmax(d)`` (lowest index on ties).
* uniforms are 24-bit integers times 2**-24, so every float32 value lies in
  [0, 1) exactly.  Column t < K is the acceptance draw r_t of position t,
  column K is the single draw u used for the replacement or bonus token.
* the ragged workload also draws, per batch row, how many drafted tokens
  the row verifies: K_b uniform in {0, ..., K} (its draw u is column K_b).
* the tree workload drafts a fixed tree per row (branching 3, 2, 1, 1 by
  depth: 21 nodes, parents listed before children); its target slots are
  N(0, 2) logits (slot 0 after the context, slot i + 1 after node i).  The
  first child of every slot takes that slot's argmax with probability 0.75,
  and every other node takes a uniform token.
"""
from __future__ import annotations

import dataclasses
import os
import sys
from typing import Iterable, Sequence

import numpy as np

# purposes of the independent streams
_S_TEMP, _S_TARGET, _S_DRAFT, _S_TOKENS, _S_UNIF, _S_PEAKS, _S_KROW, _S_TREE = range(8)

WORKLOADS = {
    # B=1, K=4, V=1000 float32; target ~ N(0, 2.0); draft = target + N(0, 0.5);
    # T = 1.0; tokens sampled from q.
    "tiny_stochastic": dict(id=1, B=1, K=4, V=1000, dtype="f32"),
    # the same inputs (logits, drafted tokens, uniforms), verified at T = 0
    "tiny_greedy": dict(id=1, B=1, K=4, V=1000, dtype="f32"),
    # B=32, K=5, V=32000 bf16; target ~ N(0, 3.0) plus one +8 peak per row;
    # draft = target + N(0, 1.0); tokens = argmax(draft); T = 0.
    "greedy_batch": dict(id=2, B=32, K=5, V=32000, dtype="bf16"),
    # B=64, K=4, V=128256 bf16; Zipf-like target; draft = target + N(0, s_b)
    # with s_b = (0.2, 0.6, 1.2)[b % 3]; T = 1.0; tokens sampled from q.
    "llama3_stochastic": dict(id=3, B=64, K=4, V=128256, dtype="bf16"),
    # B=256, K=8, V=152064 float32; Zipf-like target; draft = target +
    # N(0, 0.5); T_b ~ U(0.3, 1.5) with every tenth row (b % 10 == 0) greedy.
    "long_draft_mixed_t": dict(id=4, B=256, K=8, V=152064, dtype="f32"),
    # B=512, K=10, V=262144 bf16; target ~ N(0, 2.5) plus 1..4 peaks of +6;
    # draft = 0.8 target + N(0, 0.8); even rows T = 0.7, odd rows greedy.
    "large_vocab_stress": dict(id=5, B=512, K=10, V=262144, dtype="bf16"),
    # adaptive verification: the Llama-3 rows (same generator), but row b
    # verifies only its first K_b drafted tokens, K_b uniform in {0..4}.
    "llama3_ragged": dict(id=6, gen=3, B=64, K=4, V=128256, dtype="bf16", ragged=True),
    # greedy tree verification at the Llama-3 vocabulary: B=64 rows, a
    # 21-node draft tree each (K = N = 21 nodes, N + 1 target slots), bf16.
    "llama3_tree": dict(id=7, B=64, K=21, V=128256, dtype="bf16", tree=(3, 2, 1, 1)),
}

# the order of the five workloads, smallest first
ORDER = ["tiny_stochastic", "greedy_batch", "llama3_stochastic",
         "long_draft_mixed_t", "large_vocab_stress"]


@dataclasses.dataclass
class Workload:
    """One batch of verify inputs in storage form (host numpy arrays).

    ``target`` is [B, K+1, V] and ``draft`` is [B, K, V]; both are float32
    for ``dtype == "f32"`` or uint16 bf16 bit patterns for ``dtype == "bf16"``.
    """
    name: str
    B: int
    K: int
    V: int
    dtype: str
    target: np.ndarray
    draft: np.ndarray
    draft_tokens: np.ndarray   # [B, K] int32
    uniforms: np.ndarray       # [B, K+1] float32 in [0, 1)
    temperature: np.ndarray    # [B] float32, 0 = greedy row
    rows: np.ndarray           # [B] batch-row ids within the full workload
    k_per_row: np.ndarray | None = None   # [B] int32 K_b (ragged workloads only)
    parents: np.ndarray | None = None     # [B, N] int32 tree parents (tree workloads only)

    @property
    def elt(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def logit_bytes(self) -> int:
        return self.target.nbytes + self.draft.nbytes


def _rng(seed: int, wid: int, b: int, purpose: int, t: int = 0) -> np.random.Generator:
    ss = np.random.SeedSequence(seed, spawn_key=(wid, b, purpose, t))
    return np.random.Generator(np.random.PCG64(ss))


def _store(x64: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values once to the storage type."""
    f32 = x64.astype(np.float32)
    if dtype == "f32":
        return f32
    u = f32.view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def _stored_as_f64(raw: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return raw.astype(np.float64)
    return (raw.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _zipf_row(rng: np.random.Generator, V: int) -> np.ndarray:
    # logit = -1.1 * ln(rank) + N(0, 0.3), ranks 1..V in a random order
    rank = rng.permutation(V).astype(np.float64) + 1.0
    return -1.1 * np.log(rank) + rng.normal(0.0, 0.3, V)


def _temperature(name: str, seed: int, wid: int, b: int) -> float:
    if name in ("tiny_greedy", "greedy_batch"):
        return 0.0
    if name in ("tiny_stochastic", "llama3_stochastic", "llama3_ragged"):
        return 1.0
    if name == "long_draft_mixed_t":
        if b % 10 == 0:
            return 0.0
        return float(np.float32(_rng(seed, wid, b, _S_TEMP).uniform(0.3, 1.5)))
    if name == "large_vocab_stress":
        return 0.7 if b % 2 == 0 else 0.0
    raise KeyError(name)


def _row(name: str, seed: int, b: int, K: int, V: int, dtype: str):
    """Build batch row b: (target[K+1,V], draft[K,V], tokens[K], uniforms[K+1], T, K_b)."""
    wid = WORKLOADS[name]["id"]
    gen = WORKLOADS[name].get("gen", wid)   # which value recipe (the id seeds the streams)
    T = _temperature(name, seed, wid, b)
    tgt64 = np.empty((K + 1, V))
    for t in range(K + 1):
        rng = _rng(seed, wid, b, _S_TARGET, t)
        if gen == 1:
            row = rng.normal(0.0, 2.0, V)
        elif gen == 2:
            row = rng.normal(0.0, 3.0, V)
            row[_rng(seed, wid, b, _S_PEAKS, t).integers(0, V)] += 8.0
        elif gen in (3, 4):
            row = _zipf_row(rng, V)
        else:
            row = rng.normal(0.0, 2.5, V)
            pk = _rng(seed, wid, b, _S_PEAKS, t)
            n_peaks = int(pk.integers(1, 5))
            row[pk.choice(V, size=n_peaks, replace=False)] += 6.0
        tgt64[t] = row
    dr64 = np.empty((K, V))
    for t in range(K):
        rng = _rng(seed, wid, b, _S_DRAFT, t)
        if gen == 1:
            dr64[t] = tgt64[t] + rng.normal(0.0, 0.5, V)
        elif gen == 2:
            dr64[t] = tgt64[t] + rng.normal(0.0, 1.0, V)
        elif gen == 3:
            dr64[t] = tgt64[t] + rng.normal(0.0, (0.2, 0.6, 1.2)[b % 3], V)
        elif gen == 4:
            dr64[t] = tgt64[t] + rng.normal(0.0, 0.5, V)
        else:
            dr64[t] = 0.8 * tgt64[t] + rng.normal(0.0, 0.8, V)
    tgt = _store(tgt64, dtype)
    dr = _store(dr64, dtype)
    # drafted tokens: x_t ~ q_t, sampled from the *stored* draft values
    dstored = _stored_as_f64(dr, dtype)
    # the greedy tiny variant verifies the very tokens the T = 1 variant drafted
    T_draft = 1.0 if name == "tiny_greedy" else T
    tokens = np.empty(K, np.int32)
    for t in range(K):
        if T_draft == 0.0:
            tokens[t] = int(np.argmax(dstored[t]))
        else:
            U = _rng(seed, wid, b, _S_TOKENS, t).random(V)
            with np.errstate(divide="ignore"):
                g = -np.log(-np.log(U))
            tokens[t] = int(np.argmax(dstored[t] / np.float64(np.float32(T_draft)) + g))
    ints = _rng(seed, wid, b, _S_UNIF).integers(0, 1 << 24, K + 1)
    unif = (ints.astype(np.float64) * 2.0 ** -24).astype(np.float32)
    kb = int(_rng(seed, wid, b, _S_KROW).integers(0, K + 1)) if WORKLOADS[name].get("ragged") else K
    return tgt, dr, tokens, unif, np.float32(T), kb


def tree_parents(branching) -> np.ndarray:
    """Parents of a fixed tree, breadth first: every node of depth d has
    branching[d] children; -1 is the root."""
    parents = []
    level = [-1]
    for width in branching:
        nxt = []
        for p in level:
            for _ in range(width):
                parents.append(p)
                nxt.append(len(parents) - 1)
        level = nxt
    return np.asarray(parents, np.int32)


def _tree_row(name: str, seed: int, b: int, N: int, V: int, dtype: str):
    """Batch row b of a tree workload: (target[N+1,V], node tokens[N], parents[N])."""
    wid = WORKLOADS[name]["id"]
    parents = tree_parents(WORKLOADS[name]["tree"])
    assert len(parents) == N
    tgt64 = np.empty((N + 1, V))
    for s in range(N + 1):
        tgt64[s] = _rng(seed, wid, b, _S_TARGET, s).normal(0.0, 2.0, V)
    tgt = _store(tgt64, dtype)
    am = _stored_as_f64(tgt, dtype).argmax(axis=1)   # lowest index on ties
    pick = _rng(seed, wid, b, _S_TREE)
    tokens = np.empty(N, np.int32)
    first_child = {}
    for i in range(N):
        slot = 0 if parents[i] < 0 else int(parents[i]) + 1
        first = slot not in first_child
        first_child.setdefault(slot, i)
        match = pick.random() < 0.75
        rnd = int(pick.integers(0, V))
        tokens[i] = int(am[slot]) if (first and match) else rnd
    return tgt, tokens, parents


def _rows_job(args):
    name, seed, rows, K, V, dtype = args
    if WORKLOADS[name].get("tree"):
        return [_tree_row(name, seed, b, K, V, dtype) for b in rows]
    return [_row(name, seed, b, K, V, dtype) for b in rows]


def make(name: str, seed: int = 0, rows: Sequence[int] | None = None,
         workers: int | None = None) -> Workload:
    """Generate workload ``name`` with ``seed``.

    ``rows`` selects a subset of batch rows (their values are identical to
    the same rows of the full workload).  ``workers`` > 1 builds rows in a
    process pool started with ``spawn`` (safe after CUDA initialisation).
    """
    cfg = WORKLOADS[name]
    B, K, V, dtype = cfg["B"], cfg["K"], cfg["V"], cfg["dtype"]
    rows = np.arange(B) if rows is None else np.asarray(list(rows), dtype=np.int64)
    nb = len(rows)
    sdt = np.float32 if dtype == "f32" else np.uint16
    target = np.empty((nb, K + 1, V), sdt)
    draft = np.empty((nb, 0 if cfg.get("tree") else K, V), sdt)
    tokens = np.empty((nb, K), np.int32)
    unif = np.empty((nb, K + 1), np.float32)
    temp = np.empty(nb, np.float32)
    krow = np.empty(nb, np.int32)
    if workers is None:
        workers = 1
    main_file = getattr(sys.modules.get("__main__"), "__file__", None)
    if workers > 1 and not (main_file and os.path.exists(main_file)):
        workers = 1   # spawn children must re-import __main__; stdin/REPL has nothing to import
    chunks = [rows[i::workers] for i in range(workers)] if workers > 1 else [rows]
    if workers > 1 and nb > 1:
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        with ctx.Pool(workers) as pool:
            parts = pool.map(_rows_job, [(name, seed, [int(b) for b in c], K, V, dtype)
                                         for c in chunks])
    else:
        parts = [_rows_job((name, seed, [int(b) for b in rows], K, V, dtype))]
        chunks = [rows]
    pos = {int(b): i for i, b in enumerate(rows)}
    if cfg.get("tree"):
        par = np.empty((nb, K), np.int32)
        for c, part in zip(chunks, parts):
            for b, (tg, tk, pa) in zip(c, part):
                i = pos[int(b)]
                target[i], tokens[i], par[i] = tg, tk, pa
        # no draft rows, uniforms or temperatures: greedy verification of the tree
        return Workload(name, nb, K, V, dtype, target, np.empty((nb, 0, V), sdt), tokens,
                        np.zeros((nb, K + 1), np.float32), np.zeros(nb, np.float32),
                        rows.astype(np.int64), None, par)
    for c, part in zip(chunks, parts):
        for b, (tg, dr, tk, un, T, kb) in zip(c, part):
            i = pos[int(b)]
            target[i], draft[i], tokens[i], unif[i], temp[i], krow[i] = tg, dr, tk, un, T, kb
    return Workload(name, nb, K, V, dtype, target, draft, tokens, unif, temp,
                    rows.astype(np.int64), krow if cfg.get("ragged") else None)


def default_workers() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def shard_rows(B: int, rank: int, world: int) -> np.ndarray:
    """Contiguous shard of batch rows owned by ``rank`` of ``world``."""
    lo = (B * rank) // world
    hi = (B * (rank + 1)) // world
    return np.arange(lo, hi)


def custom(target: np.ndarray, draft: np.ndarray, draft_tokens: Iterable[Iterable[int]],
           uniforms: np.ndarray, temperature: np.ndarray, dtype: str = "f32",
           name: str = "custom") -> Workload:
    """Wrap hand-built float64 logits as a workload (rounded to ``dtype``)."""
    target = np.ascontiguousarray(target, np.float64)
    draft = np.ascontiguousarray(draft, np.float64)
    B, K1, V = target.shape
    return Workload(name, B, K1 - 1, V, dtype, _store(target, dtype), _store(draft, dtype),
                    np.asarray(draft_tokens, np.int32).reshape(B, K1 - 1),
                    np.asarray(uniforms, np.float32).reshape(B, K1),
                    np.asarray(temperature, np.float32).reshape(B), np.arange(B))
