"""Comparison of the CUDA path's outputs with the CPU oracle's.

TEST INFRASTRUCTURE ONLY, like the oracle itself: the tests and the CPU
baseline leg of ``bench.py`` (which reports these counts for the batch it
times) use it; the product path never does.

Rules (the GPU must meet all of them):
* greedy rows (T == 0) and error rows: accepted_len and out_tokens
  bit-exact;
* tempered rows: log p_t(x_t) and log q_t(x_t) within 1e-5 absolute at every
  drafted position; accepted_len and out_tokens identical, except on rows the
  oracle marks as ambiguous -- a decided position whose |r - p/q| is below
  1e-5, or a sampled u within 1e-5 of a CDF boundary.  Such mismatches are
  counted; they must stay below 0.1 % of the rows checked (callers that check
  few rows pass their own allowance).
* every row: 0 <= accepted_len <= K (or -1), out_tokens[:n] are the drafted
  tokens, the emitted token lies in [0, V), later slots are -1.
"""
from __future__ import annotations

import dataclasses

import numpy as np

LOGPROB_ATOL = 1e-5
MARGIN = 1e-5


@dataclasses.dataclass
class ParityReport:
    rows: int = 0
    greedy_rows: int = 0
    stochastic_rows: int = 0
    ambiguous_rows: int = 0
    mismatched_rows: int = 0
    max_logprob_err: float = 0.0
    failures: list = dataclasses.field(default_factory=list)

    def merge(self, o: "ParityReport") -> "ParityReport":
        return ParityReport(self.rows + o.rows, self.greedy_rows + o.greedy_rows,
                            self.stochastic_rows + o.stochastic_rows,
                            self.ambiguous_rows + o.ambiguous_rows,
                            self.mismatched_rows + o.mismatched_rows,
                            max(self.max_logprob_err, o.max_logprob_err),
                            self.failures + o.failures)


def _logprob_err(gpu, ref):
    """Largest |difference|; equal infinities (a -inf logit) count as exact,
    and so do positions both sides mark NaN (positions a ragged row does not
    verify); a NaN on one side only is an infinite error."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    same = (gpu == ref) | (np.isnan(gpu) & np.isnan(ref))
    with np.errstate(invalid="ignore"):
        d = np.where(same, 0.0, np.abs(gpu - ref))
    d = np.where(np.isnan(d), np.inf, d)
    return float(d.max()) if d.size else 0.0


def check_structure(accepted, out_tokens, draft_tokens, V):
    """Properties that hold for every row at any size."""
    B, K1 = out_tokens.shape
    K = K1 - 1
    bad = []
    for b in range(B):
        n = int(accepted[b])
        if n == -1:
            if not (out_tokens[b] == -1).all():
                bad.append((b, "error row with tokens"))
            continue
        if not 0 <= n <= K:
            bad.append((b, f"accepted_len {n}"))
            continue
        if not np.array_equal(out_tokens[b, :n], draft_tokens[b, :n]):
            bad.append((b, "accepted prefix differs from drafted tokens"))
        if not 0 <= out_tokens[b, n] < V:
            bad.append((b, f"emitted token {out_tokens[b, n]} out of range"))
        if not (out_tokens[b, n + 1:] == -1).all():
            bad.append((b, "padding is not -1"))
    return bad


def compare(ref, accepted, out_tokens, logp, logq, temperature, rows=None) -> ParityReport:
    """``ref`` is an oracle BatchResult over the same rows (``rows`` maps the
    oracle's row i to the GPU row rows[i]; default: identity)."""
    B = len(ref.accepted_len)
    rows = np.arange(B) if rows is None else np.asarray(rows)
    rep = ParityReport()
    for i in range(B):
        g = int(rows[i])
        rep.rows += 1
        n_ref = int(ref.accepted_len[i])
        same = (int(accepted[g]) == n_ref and np.array_equal(out_tokens[g], ref.out_tokens[i]))
        T = float(temperature[g])
        if T == 0.0 or n_ref == -1:
            rep.greedy_rows += T == 0.0
            if not same:
                rep.failures.append((g, "greedy/error row differs", int(accepted[g]), n_ref,
                                     out_tokens[g].tolist(), ref.out_tokens[i].tolist()))
            continue
        rep.stochastic_rows += 1
        if logp is not None:
            err = max(_logprob_err(logp[g], ref.logp[i]), _logprob_err(logq[g], ref.logq[i]))
            if not err <= LOGPROB_ATOL:
                rep.failures.append((g, f"log-prob error {err}"))
            rep.max_logprob_err = max(rep.max_logprob_err, float(err))
        decided = min(n_ref + 1, len(ref.ratio_margin[i]))
        ambiguous = (bool((ref.ratio_margin[i][:decided] < MARGIN).any())
                     or ref.cdf_margin[i] < MARGIN)
        rep.ambiguous_rows += int(ambiguous)
        if not same:
            rep.mismatched_rows += 1
            if not ambiguous:
                rep.failures.append((g, "tokens differ on an unambiguous row", int(accepted[g]),
                                     n_ref, out_tokens[g].tolist(), ref.out_tokens[i].tolist(),
                                     float(ref.cdf_margin[i])))
    return rep
