"""CPU oracle for the batched speculative-decoding verify-and-accept step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
links this module: only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use it.  It shares no code, tables or constants
with the CUDA path; both sides read the same seeded inputs, nothing else.

It is plain, slow float64 numpy, one batch row at a time, written from these
pages (cited by title and section):

[L25-PT] "Decodificação Especulativa e EAGLE", ai-engineering.academy,
         phase 10 lesson 25 (Portuguese).  Primary text for the rule.
[L25-VI] "Việc giải mã giả định và Eagle", aiengineeringfromscratch.com,
         phase 10 lesson 25 (the same lesson, machine-translated).
[HF-202] "IA local 202: acelere muito a geração com speculative decoding"
         (Hugging Face live stream transcript on iania.ai).
[SONAR]  "Accelerating Sonar through speculation" (Perplexity, Russian).
[AIVARO] "Как работает speculative decoding? Как выбрать draft модель?"
         (aivaro.ru answer 440).

What one row computes ([L25-PT] "A Regra de Exatidão", "Caso ganancioso",
"O Conceito / A Configuração com Dois Modelos" steps 1-4):

* p_t = softmax(target_t / T), q_t = softmax(draft_t / T) for the K drafted
  positions, p_K at the extra (bonus) position.
* left to right, with r_t ~ U(0, 1): accept x_t iff r_t < p_t(x_t) / q_t(x_t);
  at the first rejection draw the replacement from the residual
  (p_t - q_t)+ / ||(p_t - q_t)+||_1 and stop.
* if all K are accepted draw a bonus token from p_K.
* T = 0 (greedy): accept iff argmax(p_t) == x_t, else emit argmax(p_t) and stop.

Readings taken where the pages are silent, garbled or disagree (each one is
also listed in the design notes):

R1  T divides both the draft and the target logits ([L25-PT] "Desenvolva":
    the draft softmax divides by ``temperature`` and the target forward is
    given the same ``temperature``).
R2  The test is written ``r * q(x) < p(x)``.  For q(x) > 0 this is exactly
    ``r < p/q``; with q(x) == 0 (reachable only through underflow) it accepts
    iff p(x) > 0.
R3  The residual subtracts the whole vector q_t, not the scalar q_t(x_t)
    ([L25-PT] "A Regra de Exatidão" states the pointwise (p - q)+; the
    "Desenvolva" sketch subtracts the scalar q_probs[k], which is a slip and
    is not followed).
R4  A rejection draws from the residual, never from p ([AIVARO] section 2's
    pseudocode resamples from the target logits; it contradicts [L25-PT]
    and is not followed).  [AIVARO]'s "no bonus token" is not followed either.
R5  One uniform u = uniforms[K] serves the replacement or the bonus draw,
    whichever happens (the pages draw a fresh random number; equal in law).
R6  Inverse CDF: the smallest i with C_i > u * W, where C is the inclusive
    prefix sum of the weights w and W = C_{V-1}.  This never picks a
    zero-weight token.  If rounding leaves u * W >= C_{V-1}, the last index
    with w > 0 is taken.
R7  If the residual is identically zero (p == q to rounding) the replacement
    is drawn from p_t with the same u.  Exact arithmetic never gets here.
R8  Greedy rows compare against argmax of the raw target logits (T plays no
    part), ties going to the lowest index; the bonus is argmax(p_K).  Greedy
    rows read neither the draft logits nor the uniforms.
R9  accepted_len counts accepted drafted tokens (0..K); accepted_len + 1
    tokens are emitted; unused slots of out_tokens hold -1.
R10 A row whose temperature is negative, NaN, infinite or a nonzero value
    below the smallest normal float32, whose drafted token lies outside
    [0, V), or whose logit row has no finite maximum, is an error row:
    accepted_len = -1 and every out_tokens slot is -1.
R11 Logits may be -inf (probability 0); NaN and +inf are outside the
    contract (this oracle raises on them).
R13 Adaptive verification (spec_verify_ragged): row b with K_b drafted
    tokens is the fixed-K rule on its prefix, with u = uniforms[b, K_b];
    K_b outside [0, K] makes an error row.
R15 Greedy tree verification: a node is accepted iff its parent is (or is
    the root) and its token is the target argmax at the parent's slot; the
    deepest accepted node (lowest index on ties) gives the path, plus the
    argmax at its own slot.
R14 The plug step appends the n + 1 emitted tokens of a row at its current
    length, drops what would land past the buffer (the row is then marked
    clipped and its length stops at the buffer's end) and leaves error rows
    unchanged; also rows whose length lies outside the buffer or whose n
    exceeds K (not a length the verify step writes).
"""
from __future__ import annotations

import dataclasses

import numpy as np

FLT_MIN = 1.1754943508222875e-38  # smallest normal float32


def decode_logits(raw: np.ndarray, dtype: str) -> np.ndarray:
    """Stored logits -> float64.  bf16 is held as uint16 bit patterns."""
    if dtype == "f32":
        return np.asarray(raw, np.float32).astype(np.float64)
    if dtype == "bf16":
        bits = np.asarray(raw, np.uint16).astype(np.uint32) << 16
        return bits.view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def log_softmax(z: np.ndarray, T: float) -> np.ndarray:
    """log softmax(z / T) in float64 by the max-shifted log-sum-exp.

    [L25-PT] "Desenvolva": ``softmax(q_draft(state) / temperature)``.
    """
    s = z / T
    m = np.max(s)
    return s - m - np.log(np.sum(np.exp(s - m)))


def residual(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """Un-normalised residual (p - q)+ ([L25-PT] "A Regra de Exatidão")."""
    return np.maximum(p - q, 0.0)


def inverse_cdf(w: np.ndarray, u: float) -> int:
    """Smallest i with C_i > u * W (reading R6).  ``w`` must have a positive sum."""
    C = np.cumsum(w)
    W = C[-1]
    hits = np.nonzero(C > u * W)[0]
    if hits.size:
        return int(hits[0])
    return int(np.nonzero(w > 0)[0][-1])


def cdf_margin(w: np.ndarray, u: float) -> float:
    """Distance of u from the nearest CDF boundary C_i / W (boundaries 0 and 1 included)."""
    C = np.cumsum(w)
    W = C[-1]
    bounds = np.concatenate(([0.0], C / W))
    return float(np.min(np.abs(bounds - u)))


@dataclasses.dataclass
class RowResult:
    accepted_len: int
    out_tokens: np.ndarray          # [K+1] int32, -1 padded
    logp: np.ndarray                # [K] float64 log p_t(x_t) (NaN on greedy/error rows)
    logq: np.ndarray                # [K] float64 log q_t(x_t)
    ratio_margin: np.ndarray        # [K] |r_t - p_t(x_t)/q_t(x_t)| (inf where undecided)
    cdf_margin: float               # distance of u from a boundary of the sampled CDF
    mode: str                       # greedy | residual | residual_p | bonus | error


def _error_row(K: int) -> RowResult:
    nan = np.full(K, np.nan)
    return RowResult(-1, np.full(K + 1, -1, np.int32), nan, nan.copy(),
                     np.full(K, np.inf), np.inf, "error")


def _valid_temperature(T: float) -> bool:
    return bool(np.isfinite(T) and (T == 0.0 or T >= FLT_MIN))


def verify_row(target: np.ndarray, draft: np.ndarray, tokens: np.ndarray,
               uniforms: np.ndarray, T: float) -> RowResult:
    """Verify one row.

    target [K+1, V] and draft [K, V] are float64 logits; tokens [K] the
    drafted ids x_0..x_{K-1}; uniforms [K+1] = r_0..r_{K-1}, u; T >= 0.
    """
    target = np.asarray(target, np.float64)
    draft = np.asarray(draft, np.float64)
    K = len(tokens)
    V = target.shape[1]
    if np.isnan(target).any() or np.isposinf(target).any():
        raise ValueError("NaN or +inf target logits are outside the contract")
    T = float(T)
    if not _valid_temperature(T):
        return _error_row(K)
    if any(int(x) < 0 or int(x) >= V for x in tokens):
        return _error_row(K)
    if not np.isfinite(target.max(axis=1)).all():
        return _error_row(K)
    out = np.full(K + 1, -1, np.int32)
    nan = np.full(K, np.nan)
    if T == 0.0:
        # [L25-PT] "Caso ganancioso": accept iff argmax(p) == x_t, else emit
        # argmax(p) and stop; all accepted -> argmax(p_K) (reading R8).
        # np.argmax returns the first occurrence of the maximum.
        for t in range(K):
            a = int(np.argmax(target[t]))
            if a != int(tokens[t]):
                out[:t] = tokens[:t]
                out[t] = a
                return RowResult(t, out, nan, nan.copy(), np.full(K, np.inf), np.inf, "greedy")
        out[:K] = tokens
        out[K] = int(np.argmax(target[K]))
        return RowResult(K, out, nan, nan.copy(), np.full(K, np.inf), np.inf, "greedy")

    if np.isnan(draft).any() or np.isposinf(draft).any():
        raise ValueError("NaN or +inf draft logits are outside the contract")
    if not np.isfinite(draft.max(axis=1)).all():
        return _error_row(K)

    logP = np.stack([log_softmax(target[t], T) for t in range(K + 1)])
    logQ = (np.stack([log_softmax(draft[t], T) for t in range(K)]) if K else
            np.empty((0, V)))
    return accept_and_sample(logP, logQ, tokens, uniforms)


def accept_and_sample(logP: np.ndarray, logQ: np.ndarray, tokens: np.ndarray,
                      uniforms: np.ndarray) -> RowResult:
    """The rule itself, given the distributions of one row.

    logP [K+1, V] = log p_0..log p_K, logQ [K, V] = log q_0..log q_{K-1}
    (float64), tokens [K], uniforms [K+1] = r_0..r_{K-1}, u.
    [L25-PT] "A Regra de Exatidão" and "O Conceito" steps 3-4.
    """
    K = len(tokens)
    out = np.full(K + 1, -1, np.int32)
    logp = np.array([logP[t][int(tokens[t])] for t in range(K)], np.float64)
    logq = np.array([logQ[t][int(tokens[t])] for t in range(K)], np.float64)
    margin = np.full(K, np.inf)
    u = float(uniforms[K])
    # left to right, stop at the first rejection
    for t in range(K):
        x = int(tokens[t])
        r = float(uniforms[t])
        p_x = np.exp(logp[t])
        q_x = np.exp(logq[t])
        if q_x > 0:
            margin[t] = abs(r - p_x / q_x)
        if r * q_x < p_x:                      # reading R2
            continue
        p = np.exp(logP[t])
        q = np.exp(logQ[t])
        w = residual(p, q)
        mode = "residual"
        if not (w.sum() > 0):                  # reading R7
            w = p
            mode = "residual_p"
        out[:t] = tokens[:t]
        out[t] = inverse_cdf(w, u)
        return RowResult(t, out, logp, logq, margin, cdf_margin(w, u), mode)
    # all K accepted: bonus token from p_K ([L25-PT] step 4)
    pK = np.exp(logP[K])
    out[:K] = tokens
    out[K] = inverse_cdf(pK, u)
    return RowResult(K, out, logp, logq, margin, cdf_margin(pK, u), "bonus")


@dataclasses.dataclass
class BatchResult:
    accepted_len: np.ndarray        # [B] int32
    out_tokens: np.ndarray          # [B, K+1] int32
    logp: np.ndarray                # [B, K] float64
    logq: np.ndarray                # [B, K] float64
    ratio_margin: np.ndarray        # [B, K]
    cdf_margin: np.ndarray          # [B]
    mode: list


def spec_verify(target_logits, draft_logits, draft_tokens, uniforms, temperature,
                dtype: str | None = None) -> BatchResult:
    """The whole batch, one row at a time.

    With ``dtype`` given the logits are in storage form (float32, or uint16
    bf16 bit patterns) and are decoded first; otherwise they are float64.
    """
    B = len(temperature)
    K = np.asarray(draft_tokens).shape[1]
    al = np.empty(B, np.int32)
    ot = np.empty((B, K + 1), np.int32)
    lp = np.empty((B, K))
    lq = np.empty((B, K))
    rm = np.empty((B, K))
    cm = np.empty(B)
    modes = []
    for b in range(B):
        tg = target_logits[b]
        dr = draft_logits[b]
        if dtype is not None:
            tg = decode_logits(tg, dtype)
            dr = decode_logits(dr, dtype)
        res = verify_row(tg, dr, np.asarray(draft_tokens[b]), np.asarray(uniforms[b]),
                         float(temperature[b]))
        al[b], ot[b], lp[b], lq[b] = res.accepted_len, res.out_tokens, res.logp, res.logq
        rm[b], cm[b] = res.ratio_margin, res.cdf_margin
        modes.append(res.mode)
    return BatchResult(al, ot, lp, lq, rm, cm, modes)


def spec_verify_ragged(target_logits, draft_logits, draft_tokens, uniforms, temperature,
                       k_per_row, dtype: str | None = None) -> BatchResult:
    """Adaptive verification: row b verifies only its first K_b drafted
    tokens, 0 <= K_b <= K.  The stream transcript "IA local 202: acelere
    muito a geração com speculative decoding" (44:15-45:16, "adaptive
    verification") describes validating a different number of drafted
    tokens per request.

    Reading R13: row b is the fixed-K rule on its prefix -- target rows
    0..K_b, draft rows 0..K_b-1, tokens x_0..x_{K_b-1}, acceptance draws
    r_0..r_{K_b-1} and the replacement/bonus draw u = uniforms[b, K_b]
    (the column right after its own draws).  Outputs keep the padded K
    layout: out_tokens slots after the emitted ones are -1 and the
    log-probabilities of positions K_b..K-1 are NaN.  K_b outside [0, K]
    makes an error row (reading R10's convention).
    """
    B = len(temperature)
    K = np.asarray(draft_tokens).shape[1]
    k_per_row = np.asarray(k_per_row)
    al = np.empty(B, np.int32)
    ot = np.full((B, K + 1), -1, np.int32)
    lp = np.full((B, K), np.nan)
    lq = np.full((B, K), np.nan)
    rm = np.full((B, K), np.inf)
    cm = np.full(B, np.inf)
    modes = []
    for b in range(B):
        kb = int(k_per_row[b])
        if kb < 0 or kb > K:
            al[b] = -1
            modes.append("error")
            continue
        tg = target_logits[b][:kb + 1]
        dr = draft_logits[b][:kb]
        if dtype is not None:
            tg = decode_logits(tg, dtype)
            dr = decode_logits(dr, dtype)
        unif = np.asarray(uniforms[b])[:kb + 1]
        res = verify_row(tg, dr, np.asarray(draft_tokens[b])[:kb], unif, float(temperature[b]))
        al[b] = res.accepted_len
        ot[b, :kb + 1] = res.out_tokens
        lp[b, :kb], lq[b, :kb] = res.logp, res.logq
        rm[b, :kb], cm[b] = res.ratio_margin, res.cdf_margin
        modes.append(res.mode)
    return BatchResult(al, ot, lp, lq, rm, cm, modes)


@dataclasses.dataclass
class TreeResult:
    accepted_len: np.ndarray    # [B] int32: depth of the accepted path (-1 = error row)
    out_tokens: np.ndarray      # [B, N+1] int32: path tokens, then the bonus token, then -1
    accepted_nodes: np.ndarray  # [B, N] int32: node indices along the path, then -1


def verify_tree_greedy_row(target: np.ndarray, node_tokens: np.ndarray,
                           parents: np.ndarray):
    """Greedy verification of one draft tree.

    The lesson's section "Verificação de Atenção em Árvore" checks every node
    of a draft tree in one target pass, keeping the longest prefix along any
    accepted path; its exercise 4 asks that the target accept the longest
    correct branch.  The Sonar page's EAGLE section keeps the longest
    acceptable sequence and adds one token from the target.

    Reading R15: node i has token node_tokens[i] and parent parents[i]
    (-1 = the root, else an earlier node, so parents[i] < i).  target[0] is
    the slot after the context (the root) and target[i + 1] the slot after
    node i.  Node i is accepted iff its parent is the root or accepted, and
    node_tokens[i] == argmax(target[slot of its parent]) (np.argmax, lowest
    index on ties).  The deepest accepted node wins, with ties going to the
    lowest node index.  The output is the tokens along its path, then the
    bonus argmax(target[its slot]).  With no node accepted, the output is
    the root's argmax alone.  A parent outside [-1, i) or a token outside
    [0, V) makes an error row.
    Returns (depth, tokens along the path + bonus, nodes along the path).
    """
    target = np.asarray(target, np.float64)
    N = len(node_tokens)
    V = target.shape[1]
    for i in range(N):
        if not (-1 <= int(parents[i]) < i) or not (0 <= int(node_tokens[i]) < V):
            return -1, [], []
    if not np.isfinite(target.max(axis=1)).all():
        return -1, [], []
    am = [int(np.argmax(target[s])) for s in range(N + 1)]
    accepted = np.zeros(N, bool)
    depth = np.zeros(N, np.int64)
    for i in range(N):                       # parents come first
        p = int(parents[i])
        ok_parent = p < 0 or accepted[p]
        slot = 0 if p < 0 else p + 1
        accepted[i] = ok_parent and int(node_tokens[i]) == am[slot]
        depth[i] = 1 if p < 0 else depth[p] + 1
    best = -1
    for i in range(N):
        if accepted[i] and (best < 0 or depth[i] > depth[best]):
            best = i
    if best < 0:
        return 0, [am[0]], []
    path = []
    i = best
    while i >= 0:
        path.append(i)
        i = int(parents[i])
    path.reverse()
    return len(path), [int(node_tokens[i]) for i in path] + [am[best + 1]], path


def verify_tree_greedy(target_logits, node_tokens, parents, dtype: str | None = None) -> TreeResult:
    """The whole batch: target_logits [B, N+1, V], node_tokens and parents [B, N]."""
    B, N = np.asarray(node_tokens).shape
    al = np.empty(B, np.int32)
    ot = np.full((B, N + 1), -1, np.int32)
    nodes = np.full((B, N), -1, np.int32)
    for b in range(B):
        tg = target_logits[b]
        if dtype is not None:
            tg = decode_logits(tg, dtype)
        d, toks, path = verify_tree_greedy_row(tg, np.asarray(node_tokens[b]), np.asarray(parents[b]))
        al[b] = d
        ot[b, :len(toks)] = toks
        nodes[b, :len(path)] = path
    return TreeResult(al, ot, nodes)


@dataclasses.dataclass
class PlugResult:
    tokens: np.ndarray       # [B, max_len] int32
    seq_len: np.ndarray      # [B] int32
    last_token: np.ndarray   # [B] int32 (unchanged where nothing was appended)
    clipped: np.ndarray      # [B] bool: the row's tokens did not all fit


def plug(accepted_len, out_tokens, tokens, seq_len, last_token=None) -> PlugResult:
    """Write each row's emitted tokens into its sequence and advance its length,
    on the device, so the next step needs no GPU-to-CPU read of the accepted
    lengths ("Accelerating Sonar through speculation", the single-token MTP
    schedule: once the target's input tokens are shifted, a kernel plugs the
    next target tokens into their places; the accepted count otherwise forces
    a GPU-to-CPU sync).

    Reading R14: row b with accepted_len n >= 0 appends out_tokens[b, 0..n]
    (n + 1 tokens) at tokens[b, L..L+n], L = seq_len[b], and sets seq_len[b]
    to L + n + 1 and last_token[b] to out_tokens[b, n].  Tokens that would
    land at or past max_len are dropped, seq_len stops at max_len and the row
    is marked clipped.  An error row (n = -1), or a row whose length lies
    outside [0, max_len], changes nothing; so does n > K (out_tokens has K + 1
    columns, so such an n is not a length the verify step writes).
    """
    tokens = np.array(tokens, np.int32, copy=True)
    seq_len = np.array(seq_len, np.int32, copy=True)
    B, max_len = tokens.shape
    last = (np.full(B, -1, np.int32) if last_token is None
            else np.array(last_token, np.int32, copy=True))
    clipped = np.zeros(B, bool)
    for b in range(B):
        n = int(accepted_len[b])
        if n < 0 or n >= np.shape(out_tokens)[1]:
            continue
        L = int(seq_len[b])
        if L < 0 or L > max_len:
            continue                           # a length outside the buffer: left unchanged
        for i in range(n + 1):
            if L + i < max_len:
                tokens[b, L + i] = out_tokens[b, i]
            else:
                clipped[b] = True
        seq_len[b] = min(L + n + 1, max_len)
        last[b] = out_tokens[b, n]
    return PlugResult(tokens, seq_len, last, clipped)


def expected_tokens_closed_form(alpha: float, K: int) -> float:
    """E[tokens per verify] = (1 - alpha^(K+1)) / (1 - alpha) ([L25-PT] "Aceleração Esperada")."""
    if alpha == 1.0:
        return float(K + 1)
    return (1.0 - alpha ** (K + 1)) / (1.0 - alpha)
