"""Plain fp64 CPU oracle for batched speculative-decoding verification (accept-or-resample).

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this module. The GPU library never imports, links or calls it, and the two share no code.

What it computes, and where the pages define it (page title, then section):

* [R] "Speculative decoding", rayaq.ca ml-models:
  - Mechanics, One round, steps 3-5: left-to-right accept while u < min(1, p(x)/q(x)); on the first
    rejection a replacement drawn from max(0, p - q) / sum max(0, p - q); a bonus token from p at
    position gamma + 1 when every draft survives.
  - Why the output is exactly the target's: alpha = sum_x min(p(x), q(x)); temperature applied to
    both p and q before the test.
  - The greedy case: keep drafts while they equal the target's argmax, replace the first mismatch by
    the argmax, add the bonus argmax when all match.
  - Implementation: p rows = softmax(target logits / temp), q rows = softmax(draft logits / temp).
* [B] "Inference: distillation and speculative decoding", brunomaga.github.io:
  - Draft-model speculative decoding: the same two rules (that page names the draft distribution p
    and the target q; this module uses p = target, q = draft throughout).
  - Knowledge distillation: the temperature softmax.
* [C] "Speculative decoding", cgnarendiran.github.io blog, The correction that makes it exact:
  the accept probability and the normalised residual.
* One-hot drafts ([B] Draft-model speculative decoding, the greedy-drafter special case):
  ``oracle_verify_onehot`` is the same verification with q_i = [v == x_i].
* Greedy tree verification ([B] Medusa: a tree of candidates, the longest accepted path):
  ``oracle_tree_greedy``.
* Top-k / top-p filtering before the test ([R] Why the output is exactly the target's):
  ``filtered_softmax`` and the ``top_k`` / ``top_p`` arguments of ``verify_row`` / ``oracle_verify``.
* The cache after a round ([R] Verification attention and the cache): ``kv_rollback``.

Parity status: every function below is pinned by the tests in ``tests/test_oracle.py`` and
``tests/test_montecarlo.py`` (page-printed worked examples, closed forms, identities, an exact
rational-arithmetic restatement and Monte-Carlo statistics). No function here is "parity unpinned".

Readings where the pages leave a step open (each repeated in the design notes):

* Which uniform drives what: ``u[b, i]`` (i < gamma_b) the accept test at position i, ``u[b, G]``
  the residual draw, ``u[b, G + 1]`` the bonus draw, with G = gamma_max (fixed columns).
* The library draw (torch.multinomial) is replaced by an inverse CDF in index order with a strict
  ``>``: token j = min{ j : sum_{v <= j} w_v > u * sum_v w_v }. Zero-weight tokens are never chosen.
  If rounding leaves no prefix above the threshold, the last token with w > 0 is taken.
* A residual with zero total mass at a rejection (impossible in exact arithmetic) falls back to a
  bonus-style draw from that position's p with ``u[b, G]``.
* q(x) = 0 for a drafted x gives ratio 1 (accept) when p(x) > 0, and ratio 0 (reject) when
  p(x) = 0 as well.
* Greedy rows are the rows with temperature exactly 0. Argmax ties go to the lowest index. Greedy
  alpha_i = [x_i == g_i], p(x_i) = [x_i == g_i], q(x_i) = 1 (one-hot p and one-hot drafter).
* alpha_i, p_i(x_i), q_i(x_i) are reported for every i < gamma_b, also after the first rejection;
  0 for padding positions i >= gamma_b.
* The bonus row of row b is target position gamma_b (ragged lengths), not gamma_max.
* Row errors (all outputs of the row -1 / 0): draft_len outside [0, G]; temperature NaN, negative,
  infinite or in (0, FLT_MIN); a drafted token outside [0, V) at i < gamma_b; for sampled rows a
  used uniform outside [0, 1); a read logit row holding NaN or +inf, or holding only -inf.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

MARGIN = 1e-5           # decision margin of the parity rule (absolute on u, relative on the CDF)
FLT_MIN = np.float64(np.finfo(np.float32).tiny)   # smallest normal fp32, lower bound of a sampled T


# ----------------------------------------------------------------------------------------------
# Single-position building blocks
# ----------------------------------------------------------------------------------------------

def temperature_softmax(z, T):
    """softmax(z / T) in fp64 ([R] Implementation: softmax of logits / temp for both models;
    [B] Knowledge distillation: the temperature softmax). The stored logits widen to fp64 exactly.
    -inf logits get probability 0."""
    y = np.asarray(z, dtype=np.float64) / np.float64(T)
    m = np.max(y)
    e = np.exp(y - m)
    return e / np.sum(e)


def filtered_softmax(z, T, top_k=0, top_p=1.0):
    """The distribution the rule is given after top-k and top-p filtering ([R] Why the output is
    exactly the target's: temperature, top-p and any penalties are applied to p and q before the
    test). In order: softmax(z / T); top-k keeps every token whose logit is not below the k-th
    largest (ties at the boundary all kept; top_k <= 0 or >= V keeps all); top-p, on the renormalised
    top-k distribution, keeps a token when the mass of the tokens with a strictly larger logit is
    below top_p (so ties go together and the largest logit is always kept; top_p >= 1 keeps all);
    the kept probabilities are renormalised. Returns (probabilities, top-p margin): the margin is the
    distance from top_p to the nearest cumulative mass at a logit boundary (1.0 without top-p)."""
    z = np.asarray(z, dtype=np.float64)
    p = temperature_softmax(z, T)
    V = z.shape[0]
    keep = np.ones(V, dtype=bool)
    if 0 < top_k < V:
        kth = np.sort(z)[::-1][top_k - 1]
        keep &= z >= kth
    pk = np.where(keep, p, 0.0)
    pk = pk / np.sum(pk)
    margin = 1.0
    if np.float64(top_p) < 1.0:
        levels = np.unique(z[keep])[::-1]                 # distinct kept logits, largest first
        above = 0.0
        keep_p = np.zeros(V, dtype=bool)
        margin = abs(np.float64(top_p))
        for lv in levels:
            grp = keep & (z == lv)
            if above < np.float64(top_p):
                keep_p |= grp
            above += np.sum(pk[grp])
            margin = min(margin, abs(above - np.float64(top_p)))
        keep &= keep_p
        pk = np.where(keep, pk, 0.0)
        pk = pk / np.sum(pk)
    return pk, margin


def accept_ratio(p_x, q_x):
    """min(1, p(x)/q(x)) ([R] One round, step 3; [C] The correction that makes it exact).
    q(x) = 0 (a token the drafter gave no mass, e.g. a -inf draft logit) reads as ratio 1 when
    p(x) > 0 (p >= q is always kept) and as ratio 0 when p(x) = 0 too: a token the target gives no
    mass is never emitted ([R] The output distribution is exactly the target's)."""
    if q_x <= 0.0:
        return 1.0 if p_x > 0.0 else 0.0
    return min(1.0, p_x / q_x)


def residual_weights(p, q):
    """max(0, p - q), unnormalised ([R] One round, step 4; [C] residual numerator)."""
    return np.maximum(0.0, p - q)


def inverse_cdf(w, u):
    """Token j = min{ j : sum_{v <= j} w_v > u * W } with W the running total at the end; index
    order, strict '>'. Stands in for the pages' library draw from the normalised weights w / W
    ([R] Implementation, torch.multinomial). Overrun by rounding takes the last token with w > 0."""
    c = np.cumsum(w)
    t = u * c[-1]
    hit = np.flatnonzero(c > t)
    if hit.size:
        return int(hit[0])
    return int(np.flatnonzero(w > 0)[-1])


def admissible_draws(w, u, eps=MARGIN):
    """Every token whose CDF interval [C_{j-1}, C_j] comes within eps * W of the threshold u * W.
    The draw is fixed (a single admissible token) when the threshold is farther than eps * W from
    every interval boundary. Returns (sorted token list, gap), gap = distance of the threshold to the
    nearest boundary of the chosen token's interval, divided by W."""
    c = np.cumsum(w)
    W = c[-1]
    t = u * W
    lo = np.concatenate(([0.0], c[:-1]))
    adm = np.flatnonzero((lo <= t + eps * W) & (c >= t - eps * W))
    j = inverse_cdf(w, u)
    gap = min(t - lo[j], c[j] - t) / W if W > 0 else 0.0
    last_pos = int(np.flatnonzero(w > 0)[-1])
    toks = set(int(a) for a in adm)
    if t >= W - eps * W:           # the overrun rule may apply within the margin
        toks.add(last_pos)
    toks.add(j)
    return sorted(toks), gap


def greedy_argmax(z):
    """Target argmax on the stored logits, lowest index on ties ([B] Draft-model speculative decoding,
    greedy rule; [R] The greedy case)."""
    return int(np.argmax(np.asarray(z, dtype=np.float64)))


# ----------------------------------------------------------------------------------------------
# Row validity (host-visible data errors)
# ----------------------------------------------------------------------------------------------

def _bad_logits(z):
    z = np.asarray(z, dtype=np.float64)
    return bool(np.any(np.isnan(z)) or np.any(z == np.inf) or np.all(z == -np.inf))


def row_is_valid(zt, zd, x, gamma_b, T, u, G, V):
    """Applies the row-error rules listed in the module docstring. zt: [G+1, V], zd: [G, V]."""
    if not (0 <= gamma_b <= G):
        return False
    T = np.float64(T)
    if np.isnan(T) or T < 0 or np.isinf(T) or (0 < T < FLT_MIN):
        return False
    greedy = T == 0
    for i in range(gamma_b):
        if not (0 <= int(x[i]) < V):
            return False
    if not greedy:
        used = [u[i] for i in range(gamma_b)] + [u[G], u[G + 1]]
        for uu in used:
            uu = np.float64(uu)
            if not (0.0 <= uu < 1.0):
                return False
    for i in range(gamma_b + 1):
        if _bad_logits(zt[i]):
            return False
    if not greedy:
        for i in range(gamma_b):
            if _bad_logits(zd[i]):
                return False
    return True


# ----------------------------------------------------------------------------------------------
# One row
# ----------------------------------------------------------------------------------------------

@dataclass
class RowResult:
    tokens: list            # emitted tokens (k accepted drafts + one correction or bonus), or [] on error
    k: int                  # accepted drafts, -1 on error
    alpha: np.ndarray       # [G]
    p_draft: np.ndarray     # [G]
    q_draft: np.ndarray     # [G]
    valid: bool = True
    greedy: bool = False
    ratio: np.ndarray = None        # [gamma_b] min(1, p/q) (sampled rows)
    margin: np.ndarray = None       # [gamma_b] |u_i - r_i| (sampled rows)
    outcomes: dict = field(default_factory=dict)   # legit k -> admissible final tokens (diagnostics)
    exact: bool = True              # True when the only legit outcome is (k, tokens[-1])
    final_gap: float = 1.0
    filter_margin: float = 1.0      # top-p: nearest cumulative boundary to top_p (1.0 without)


def verify_row(zt, zd, x, gamma_b, T, u, G, diagnostics=False, eps=MARGIN, top_k=0, top_p=1.0):
    """One row of the batch: the round's verification half ([R] One round steps 3-5 and
    Implementation, after the target pass; [R] The greedy case for T == 0).

    zt: [G+1, V] target logits, zd: [G, V] draft logits, x: [G] drafted tokens, u: [G+2] uniforms.
    top_k, top_p: the row's filtering, applied to p and q alike (see filtered_softmax; sampled rows).
    """
    V = np.asarray(zt).shape[-1]
    alpha = np.zeros(G)
    pd = np.zeros(G)
    qd = np.zeros(G)
    if not row_is_valid(zt, zd, x, gamma_b, T, u, G, V):
        return RowResult([], -1, alpha, pd, qd, valid=False)
    if np.float64(T) != 0.0 and not np.float64(top_p) > 0.0:
        # A nucleus of no mass keeps nothing: a sampled row asking for it has no distribution.
        return RowResult([], -1, alpha, pd, qd, valid=False)

    if np.float64(T) == 0.0:
        # Greedy: keep drafts while they equal the target argmax; the correction or bonus is the argmax.
        g = [greedy_argmax(zt[i]) for i in range(gamma_b + 1)]
        for i in range(gamma_b):
            hit = int(x[i]) == g[i]
            alpha[i] = 1.0 if hit else 0.0
            pd[i] = 1.0 if hit else 0.0
            qd[i] = 1.0
        k = 0
        while k < gamma_b and int(x[k]) == g[k]:
            k += 1
        toks = [int(x[i]) for i in range(k)] + [g[k]]
        res = RowResult(toks, k, alpha, pd, qd, greedy=True)
        res.outcomes = {k: [g[k]]}
        return res

    # Sampled row. Target p_i and draft q_i at every verified position i < gamma_b, alpha_i for each.
    ratio = np.zeros(gamma_b)
    margin = np.zeros(gamma_b)
    p_rows, q_rows = [], []
    fmargin = 1.0

    def dist(z):
        nonlocal fmargin
        w, m = filtered_softmax(z, T, top_k, top_p)
        fmargin = min(fmargin, m)
        return w

    for i in range(gamma_b):
        p = dist(zt[i])
        q = dist(zd[i])
        p_rows.append(p)
        q_rows.append(q)
        xi = int(x[i])
        pd[i], qd[i] = p[xi], q[xi]
        alpha[i] = np.sum(np.minimum(p, q))          # [R] Why the output is exactly the target's
        ratio[i] = accept_ratio(p[xi], q[xi])
        margin[i] = abs(np.float64(u[i]) - ratio[i])

    # Accept left to right, stop at the first rejection ([R] One round, step 3).
    k = 0
    while k < gamma_b and np.float64(u[k]) < ratio[k]:
        k += 1

    def final_draw(kk):
        """The token after kk accepted drafts, and its weights and uniform."""
        if kk < gamma_b:
            w = residual_weights(p_rows[kk], q_rows[kk])      # [R] One round, step 4
            uu = np.float64(u[G])
            if not np.sum(w) > 0.0:                           # zero residual mass: draw from p
                w = p_rows[kk]
        else:
            w = p_bonus                                        # [R] One round, step 5 (bonus)
            uu = np.float64(u[G + 1])
        return w, uu

    p_bonus = dist(zt[gamma_b])

    w, uu = final_draw(k)
    j = inverse_cdf(w, uu)
    res = RowResult([int(x[i]) for i in range(k)] + [j], k, alpha, pd, qd,
                    ratio=ratio, margin=margin)
    res.filter_margin = fmargin
    if diagnostics:
        # Every accept count reachable when decisions within eps of their threshold may go either way,
        # and for each the tokens whose CDF interval lies within eps of the draw's threshold.
        legit = []
        for kk in range(gamma_b + 1):
            if all(np.float64(u[i]) < ratio[i] + eps for i in range(kk)) and \
                    (kk == gamma_b or np.float64(u[kk]) >= ratio[kk] - eps):
                legit.append(kk)
        for kk in legit:
            ww, uk = final_draw(kk)
            adm, gap = admissible_draws(ww, uk, eps)
            res.outcomes[kk] = adm
            if kk == k:
                res.final_gap = gap
        res.exact = legit == [k] and res.outcomes[k] == [j]
    return res


# ----------------------------------------------------------------------------------------------
# The batch
# ----------------------------------------------------------------------------------------------

@dataclass
class BatchResult:
    out_tokens: np.ndarray       # [B, G+1] int32, -1 padding
    out_num_emitted: np.ndarray  # [B] int32, k+1 or -1
    out_alpha: np.ndarray        # [B, G] fp64
    out_p_draft: np.ndarray      # [B, G] fp64
    out_q_draft: np.ndarray      # [B, G] fp64
    rows: list                   # RowResult per row (diagnostics)


def oracle_verify(target_logits, draft_logits, draft_tokens, draft_len, temperature, uniforms,
                  rows=None, diagnostics=False, eps=MARGIN, top_k=None, top_p=None):
    """Batched verification, one row at a time in plain loops.

    target_logits [B, G+1, V], draft_logits [B, G, V] (any float dtype holding the stored values),
    draft_tokens [B, G] int, draft_len [B] int or None (all G), temperature [B] fp32 (0 = greedy),
    uniforms [B, G+2] fp32. ``rows`` restricts the work to a subset of rows (others stay -1).
    """
    target_logits = np.asarray(target_logits)
    B, G1, V = target_logits.shape
    G = G1 - 1
    if draft_len is None:
        draft_len = np.full(B, G, dtype=np.int64)
    out_tokens = np.full((B, G + 1), -1, dtype=np.int32)
    out_num = np.full(B, -1, dtype=np.int32)
    out_alpha = np.zeros((B, G))
    out_p = np.zeros((B, G))
    out_q = np.zeros((B, G))
    results = [None] * B
    for b in (range(B) if rows is None else rows):
        zd = draft_logits[b] if draft_logits is not None else np.zeros((G, V))
        r = verify_row(target_logits[b], zd, draft_tokens[b], int(draft_len[b]),
                       np.float32(temperature[b]), uniforms[b], G, diagnostics=diagnostics, eps=eps,
                       top_k=0 if top_k is None else int(top_k[b]),
                       top_p=1.0 if top_p is None else np.float64(np.float32(top_p[b])))
        results[b] = r
        if r.valid:
            out_tokens[b, :len(r.tokens)] = r.tokens
            out_num[b] = len(r.tokens)
            out_alpha[b] = r.alpha
            out_p[b] = r.p_draft
            out_q[b] = r.q_draft
    return BatchResult(out_tokens, out_num, out_alpha, out_p, out_q, results)


def oracle_verify_rows(row_source, draft_tokens, draft_len, temperature, uniforms, G, V, rows,
                       threads=1, diagnostics=False, eps=MARGIN):
    """oracle_verify over the listed rows only, several rows at a time in a pool of threads (numpy
    releases the interpreter lock inside its array operations). Each row is still verify_row, the
    plain loop above: the threads change where rows run, not what is computed.

    row_source(b) -> (zt [G+1, V], zd [G, V]) gives a row's stored logits as float arrays; it is
    called from the pool's threads. Returns a BatchResult of B = len(draft_len) rows whose
    unlisted rows stay -1 / 0 (rows[b] None)."""
    from concurrent.futures import ThreadPoolExecutor
    B = len(draft_len)
    out_tokens = np.full((B, G + 1), -1, dtype=np.int32)
    out_num = np.full(B, -1, dtype=np.int32)
    out_alpha = np.zeros((B, G))
    out_p = np.zeros((B, G))
    out_q = np.zeros((B, G))
    results = [None] * B

    def one(b):
        zt, zd = row_source(b)
        return b, verify_row(zt, zd, draft_tokens[b], int(draft_len[b]), np.float32(temperature[b]),
                             uniforms[b], G, diagnostics=diagnostics, eps=eps)

    if threads <= 1:
        done = map(one, rows)
    else:
        pool = ThreadPoolExecutor(max_workers=threads)
        done = pool.map(one, rows)
    try:
        for b, r in done:
            results[b] = r
            if r.valid:
                out_tokens[b, :len(r.tokens)] = r.tokens
                out_num[b] = len(r.tokens)
                out_alpha[b] = r.alpha
                out_p[b] = r.p_draft
                out_q[b] = r.q_draft
    finally:
        if threads > 1:
            pool.shutdown()
    return BatchResult(out_tokens, out_num, out_alpha, out_p, out_q, results)


# ----------------------------------------------------------------------------------------------
# One-hot drafts (a greedy drafter): q_i = [v == x_i]
# ----------------------------------------------------------------------------------------------

def onehot_draft_logits(x, G, V):
    """Draft logits whose temperature softmax is one-hot at the drafted token: -inf everywhere and 0
    at x_i ([B] Draft-model speculative decoding: greedy drafts are the special case of a one-hot
    draft distribution). A drafted token outside [0, V) leaves its row all -inf (the row check
    reports the token first)."""
    zd = np.full((G, V), -np.inf)
    for i in range(G):
        xi = int(x[i])
        if 0 <= xi < V:
            zd[i, xi] = 0.0
    return zd


def oracle_verify_onehot(target_logits, draft_tokens, draft_len, temperature, uniforms,
                         rows=None, diagnostics=False, eps=MARGIN):
    """Verification of one-hot drafts: oracle_verify with q_i = [v == x_i] at every drafted position
    (built row by row). With that q the rule keeps x with probability min(1, p(x)/1) = p(x), gives
    alpha = sum min(p, q) = p(x), and draws a replacement from max(0, p - q), which is p without x
    ([B] Draft-model speculative decoding)."""
    target_logits = np.asarray(target_logits)
    B, G1, V = target_logits.shape
    G = G1 - 1
    if draft_len is None:
        draft_len = np.full(B, G, dtype=np.int64)
    out_tokens = np.full((B, G + 1), -1, dtype=np.int32)
    out_num = np.full(B, -1, dtype=np.int32)
    out_alpha = np.zeros((B, G))
    out_p = np.zeros((B, G))
    out_q = np.zeros((B, G))
    results = [None] * B
    for b in (range(B) if rows is None else rows):
        zd = onehot_draft_logits(draft_tokens[b], G, V)
        r = verify_row(target_logits[b], zd, draft_tokens[b], int(draft_len[b]),
                       np.float32(temperature[b]), uniforms[b], G, diagnostics=diagnostics, eps=eps)
        results[b] = r
        if r.valid:
            out_tokens[b, :len(r.tokens)] = r.tokens
            out_num[b] = len(r.tokens)
            out_alpha[b] = r.alpha
            out_p[b] = r.p_draft
            out_q[b] = r.q_draft
    return BatchResult(out_tokens, out_num, out_alpha, out_p, out_q, results)


# ----------------------------------------------------------------------------------------------
# Greedy tree verification (Medusa-style candidate trees)
# ----------------------------------------------------------------------------------------------

@dataclass
class TreeResult:
    path: np.ndarray        # [B, N] node indices of the longest accepted path, root first, -1 padding
    path_len: np.ndarray    # [B] nodes on the path (>= 1), -1 on a row error
    tokens: np.ndarray      # [B, N+1] tokens of the path nodes, then the target's next token, -1 padding
    pred: np.ndarray        # [B, N] target argmax at every node (-1 beyond the row's nodes or on error)


def tree_row_is_valid(zt, tok, par, n, N, V):
    """Row errors of a tree row: size outside [1, N]; the root's parent not -1; a parent outside
    [0, node) for any other node; a node token outside [0, V); a node's logit row with NaN or +inf,
    or only -inf."""
    if not (1 <= n <= N):
        return False
    if int(par[0]) != -1:
        return False
    for i in range(1, n):
        if not (0 <= int(par[i]) < i):
            return False
    for i in range(n):
        if not (0 <= int(tok[i]) < V):
            return False
        if _bad_logits(zt[i]):
            return False
    return True


def oracle_tree_greedy(target_logits, tree_tokens, tree_parents, tree_size=None):
    """Greedy verification of a tree of candidates, one row at a time ([B] "Inference: distillation
    and speculative decoding" -- Medusa: the candidates form a tree verified in one target pass; the
    root is the target's own next token; a node is accepted when its parent is accepted and its
    token equals the target's argmax after its parent; the longest accepted path is kept, and the
    target's argmax after the path's last node is the next token).

    target_logits [B, N, V] (the target's logits at every node), tree_tokens [B, N], tree_parents
    [B, N] (-1 at the root, parents before children), tree_size [B] or None (all N). Argmax ties go
    to the lowest index; among the deepest accepted nodes the lowest node index ends the path."""
    target_logits = np.asarray(target_logits)
    B, N, V = target_logits.shape
    if tree_size is None:
        tree_size = np.full(B, N, dtype=np.int64)
    path = np.full((B, N), -1, dtype=np.int32)
    plen = np.full(B, -1, dtype=np.int32)
    toks = np.full((B, N + 1), -1, dtype=np.int32)
    pred = np.full((B, N), -1, dtype=np.int32)
    for b in range(B):
        n = int(tree_size[b])
        tok, par = tree_tokens[b], tree_parents[b]
        if not tree_row_is_valid(target_logits[b], tok, par, n, N, V):
            continue
        g = [greedy_argmax(target_logits[b, i]) for i in range(n)]
        accepted = {0: 1}                 # node -> nodes on its path from the root
        best = 0
        for i in range(1, n):
            pi = int(par[i])
            if pi in accepted and int(tok[i]) == g[pi]:
                accepted[i] = accepted[pi] + 1
                if accepted[i] > accepted[best]:
                    best = i
        nodes = [best]
        while nodes[-1] != 0:
            nodes.append(int(par[nodes[-1]]))
        nodes.reverse()
        L = len(nodes)
        path[b, :L] = nodes
        plen[b] = L
        toks[b, :L] = [int(tok[j]) for j in nodes]
        toks[b, L] = g[best]
        pred[b, :n] = g
    return TreeResult(path, plen, toks, pred)


# ----------------------------------------------------------------------------------------------
# KV-cache rollback after a round
# ----------------------------------------------------------------------------------------------

def kv_rollback(prefix_len, draft_len, num_emitted, drafter_len, G):
    """New cache lengths after a verified round, one row at a time ([R] Verification attention and
    the cache: keep the first n + k + 1 entries of the target's cache, the prefix, the last token
    and the accepted drafts; the drafter's cache is rolled back the same way, never beyond what it
    holds). Returns (target_len, drafter_len, dropped) with dropped[b] = (first, end) entries of the
    target cache that the round wrote and no longer keeps (end = n + gamma_b + 1). A row error
    (num_emitted < 1) commits nothing."""
    B = len(prefix_len)
    target = np.zeros(B, dtype=np.int64)
    drafter = np.zeros(B, dtype=np.int64)
    dropped = []
    for b in range(B):
        n = int(prefix_len[b])
        g = G if draft_len is None else min(max(int(draft_len[b]), 0), G)
        e = int(num_emitted[b])
        keep = n + e if e >= 1 else n          # e = k + 1
        target[b] = keep
        d = keep if drafter_len is None else int(drafter_len[b])
        drafter[b] = min(d, keep)
        dropped.append((keep, n + g + 1))
    return target, drafter, dropped


# ----------------------------------------------------------------------------------------------
# Drafting helper (input preparation for the small configuration, not the verification path)
# ----------------------------------------------------------------------------------------------

def sample_drafts(draft_logits, temperature, uniforms):
    """Draft tokens x_i ~ q_i by inverse CDF in fp64 ([R] One round, step 1: x_i ~ q). Greedy rows
    (T == 0) take the draft argmax ([B] DraftModel: greedy drafter). uniforms: [B, G] fp32."""
    draft_logits = np.asarray(draft_logits)
    B, G, V = draft_logits.shape
    x = np.zeros((B, G), dtype=np.int32)
    for b in range(B):
        for i in range(G):
            if np.float64(temperature[b]) == 0.0:
                x[b, i] = greedy_argmax(draft_logits[b, i])
            else:
                x[b, i] = inverse_cdf(temperature_softmax(draft_logits[b, i], temperature[b]),
                                      np.float64(uniforms[b, i]))
    return x
