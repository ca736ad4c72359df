"""Comparison of the GPU outputs against the fp64 oracle under the 1e-5 margin rule.

Rule: alpha, p(x) and q(x) within 1e-5 absolute at every verified position (exact zeros on padding).
Emitted tokens and accept counts are bit-exact on every row whose oracle decisions all lie farther
than 1e-5 from their thresholds (accept tests: |u - min(1, p/q)|; draws: the CDF gap relative to the
draw's total). A row with a decision inside the margin is a "margin row": its GPU accept count must
be one the oracle reaches when those decisions go either way, and its final token must lie in the
oracle's admissible set for that count. Greedy rows decide on raw logits and are always exact.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

TOL = 1e-5


@dataclass
class ParityReport:
    rows: int = 0
    exact_rows: int = 0
    margin_rows: int = 0
    error_rows: int = 0
    max_alpha_err: float = 0.0
    max_prob_err: float = 0.0
    positions: int = 0              # verified positions of the compared rows (sum of gamma_b + 1)
    margin_positions: int = 0       # decisions inside the margin (accept tests and final draws)
    failures: list = field(default_factory=list)

    def ok(self):
        return not self.failures

    def merge(self, other):
        for name in ("rows", "exact_rows", "margin_rows", "error_rows", "positions",
                     "margin_positions"):
            setattr(self, name, getattr(self, name) + getattr(other, name))
        self.max_alpha_err = max(self.max_alpha_err, other.max_alpha_err)
        self.max_prob_err = max(self.max_prob_err, other.max_prob_err)
        self.failures += other.failures
        return self

    def as_dict(self):
        return {"rows_checked": self.rows, "exact_rows": self.exact_rows,
                "margin_rows": self.margin_rows, "error_rows": self.error_rows,
                "positions_checked": self.positions, "margin_positions": self.margin_positions,
                "max_abs_alpha_err": self.max_alpha_err, "max_abs_prob_err": self.max_prob_err,
                "failures": len(self.failures)}

    def __str__(self):
        return (f"rows={self.rows} exact={self.exact_rows} margin={self.margin_rows} "
                f"error_rows={self.error_rows} positions={self.positions} "
                f"margin_positions={self.margin_positions} max|dalpha|={self.max_alpha_err:.2e} "
                f"max|dp|={self.max_prob_err:.2e} failures={self.failures[:5]}")


def compare(oracle, gpu_tokens, gpu_num, gpu_alpha, gpu_p, gpu_q, draft_tokens, draft_len,
            rows=None, tol=TOL) -> ParityReport:
    """oracle: BatchResult from oracle_verify(..., diagnostics=True); gpu_*: numpy arrays."""
    rep = ParityReport()
    B = gpu_num.shape[0]
    G = gpu_alpha.shape[1] if gpu_alpha is not None else gpu_tokens.shape[1] - 1
    for b in (range(B) if rows is None else rows):
        r = oracle.rows[b]
        rep.rows += 1
        if not r.valid:
            rep.error_rows += 1
            if gpu_num[b] != -1 or (gpu_tokens[b] != -1).any():
                rep.failures.append((b, "expected row error", int(gpu_num[b])))
            if gpu_alpha is not None and (gpu_alpha[b] != 0).any():
                rep.failures.append((b, "alpha not zeroed on error row"))
            continue
        gb = int(draft_len[b])
        rep.positions += gb + 1
        if r.margin is not None:
            rep.margin_positions += int(np.sum(r.margin < tol)) + int(r.final_gap < tol)
        if gpu_num[b] < 1:
            rep.failures.append((b, "gpu row error", int(gpu_num[b])))
            continue
        for name, g_arr, o_arr in (("alpha", gpu_alpha, oracle.out_alpha),
                                   ("p", gpu_p, oracle.out_p_draft), ("q", gpu_q, oracle.out_q_draft)):
            if g_arr is None:
                continue
            d = np.abs(g_arr[b, :gb].astype(np.float64) - o_arr[b, :gb])
            m = float(d.max()) if gb else 0.0
            if name == "alpha":
                rep.max_alpha_err = max(rep.max_alpha_err, m)
            else:
                rep.max_prob_err = max(rep.max_prob_err, m)
            if m > tol:
                rep.failures.append((b, f"{name} off by {m:.3e}"))
            if (g_arr[b, gb:] != 0).any():
                rep.failures.append((b, f"{name} padding not zero"))
        k = int(gpu_num[b]) - 1
        toks = gpu_tokens[b]
        if (toks[k + 1:] != -1).any():
            rep.failures.append((b, "token padding not -1"))
        if r.exact:
            rep.exact_rows += 1
            want = np.full(G + 1, -1, dtype=np.int64)
            want[:len(r.tokens)] = r.tokens
            if k != r.k or not np.array_equal(toks.astype(np.int64), want):
                rep.failures.append((b, "token mismatch (exact row)", r.k, r.tokens,
                                     toks[:k + 1].tolist()))
            continue
        rep.margin_rows += 1
        if k not in r.outcomes:
            rep.failures.append((b, "accept count outside margin outcomes", k, sorted(r.outcomes)))
            continue
        if not np.array_equal(toks[:k], np.asarray(draft_tokens[b, :k])):
            rep.failures.append((b, "accepted prefix differs from drafts"))
        if int(toks[k]) not in r.outcomes[k]:
            rep.failures.append((b, "final token not admissible", int(toks[k]), r.outcomes[k][:8]))
    return rep


def oracle_threads():
    """Threads for the oracle: the cores this process may run on."""
    import os
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def full_batch_parity(w, gpu, rows=None, chunk=64, threads=None, tol=TOL) -> ParityReport:
    """Every row (or the listed rows) of a workload whose logits are device tensors, compared with
    the fp64 oracle. Rows come to the host `chunk` at a time from the calling thread; the oracle
    runs each chunk's rows in a thread pool. gpu: the numpy outputs (tokens, num, alpha, p, q)."""
    from oracle.spec_verify_oracle import oracle_verify_rows
    threads = threads or oracle_threads()
    rows = list(range(w.B)) if rows is None else list(rows)
    rep = ParityReport()
    for c0 in range(0, len(rows), chunk):
        part = rows[c0:c0 + chunk]
        host = {}
        for b in part:
            host[b] = w.host_rows(b)
        o = oracle_verify_rows(lambda b: host[b], w.draft_tokens, w.draft_len, w.temperature,
                               w.uniforms, w.G, w.V, part, threads=threads, diagnostics=True,
                               eps=tol)
        rep.merge(compare(o, *gpu, w.draft_tokens, w.draft_len, rows=part, tol=tol))
        del host, o
    return rep
