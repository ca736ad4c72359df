"""Exact rational-arithmetic restatement of the accept-or-resample rule, for tiny vocabularies.

TEST INFRASTRUCTURE (same import rule as ``spec_verify_oracle``). It is a second, independent
statement of the rule in ``fractions.Fraction`` arithmetic. The tests pin it to the exact values the
pages print, and then use it to pin the fp64 oracle on tiny inputs.

Sources (page title, section):
* "Speculative decoding", rayaq.ca ml-models: Mechanics, One round (steps 1-5); Worked example
  (three-token Markov tables); A round with a rejection; The output distribution is exactly the
  target's (enumeration of a round, two-token joint); Tokens per round: exact against the formula.
* "Speculative decoding", cgnarendiran.github.io blog: The correction that makes it exact.
"""
from __future__ import annotations

from fractions import Fraction
from itertools import product


def alpha(p, q):
    """alpha = sum_x min(p(x), q(x)) (rayaq.ca, Why the output is exactly the target's)."""
    return sum(min(a, b) for a, b in zip(p, q))


def residual(p, q):
    """Normalised residual max(0, p - q) / sum max(0, p - q) (rayaq.ca, One round, step 4)."""
    w = [max(Fraction(0), a - b) for a, b in zip(p, q)]
    s = sum(w)
    return [x / s for x in w] if s > 0 else None


def accept_prob(p_x, q_x):
    """min(1, p(x)/q(x)) (rayaq.ca, One round, step 3). With q(x) = 0: 1 when p(x) > 0, 0 when
    p(x) = 0 (a token of zero target mass is never emitted: rayaq.ca, The output distribution is
    exactly the target's)."""
    if q_x == 0:
        return Fraction(1) if p_x > 0 else Fraction(0)
    return min(Fraction(1), Fraction(p_x) / Fraction(q_x))


def round_outcomes(p_next, q_next, start, gamma):
    """Exact distribution of one round from context ``start``.

    p_next(c) / q_next(c): target / draft next-token distributions after token c (Markov).
    Enumerates every draft sequence (x_1..x_gamma, x_i ~ q(. | x_{i-1})) and every accept / reject
    outcome: k accepted then a residual draw at position k+1, or all accepted then a bonus draw from
    p after x_gamma. Returns (dict emitted-sequence -> probability, list P(K = k), k = 0..gamma).
    """
    V = len(p_next(start))
    seqs = {}
    pk = [Fraction(0)] * (gamma + 1)
    for drafts in product(range(V), repeat=gamma):
        ctx = [start] + list(drafts[:-1])          # context before each draft position
        pr = Fraction(1)
        for c, x in zip(ctx, drafts):
            pr *= q_next(c)[x]
        if pr == 0:
            continue
        survive = Fraction(1)
        for k in range(gamma):
            c, x = ctx[k], drafts[k]
            a = accept_prob(p_next(c)[x], q_next(c)[x])
            rej = survive * (1 - a)
            if rej > 0:
                r = residual(p_next(c), q_next(c))
                pk[k] += pr * rej
                for y, ry in enumerate(r):
                    if ry > 0:
                        key = tuple(drafts[:k]) + (y,)
                        seqs[key] = seqs.get(key, Fraction(0)) + pr * rej * ry
            survive *= a
            if survive == 0:
                break
        if survive > 0:
            pk[gamma] += pr * survive
            for y, py in enumerate(p_next(drafts[-1])):
                if py > 0:
                    key = tuple(drafts) + (y,)
                    seqs[key] = seqs.get(key, Fraction(0)) + pr * survive * py
    return seqs, pk


def joint_first_tokens(p_next, q_next, start, gamma, n):
    """Exact joint distribution of the first n emitted tokens when rounds are chained from ``start``
    (rayaq.ca, The output distribution is exactly the target's)."""
    out = {}

    def rec(prefix, ctx, prob):
        if len(prefix) >= n:
            key = tuple(prefix[:n])
            out[key] = out.get(key, Fraction(0)) + prob
            return
        seqs, _ = round_outcomes(p_next, q_next, ctx, gamma)
        for s, ps in seqs.items():
            rec(prefix + list(s), s[-1], prob * ps)

    rec([], start, Fraction(1))
    return out


def verify_row_exact(p_rows, q_rows, drafts, u_acc, u_res, u_bonus):
    """The deterministic rule for given uniforms, in exact arithmetic.

    p_rows: gamma + 1 target distributions, q_rows: gamma draft distributions, drafts: gamma tokens,
    u_acc: gamma uniforms, u_res / u_bonus: the residual and bonus uniforms (Fractions).
    Draws use the inverse CDF in index order with a strict '>'. Returns (k, emitted tokens).
    """
    gamma = len(drafts)
    k = 0
    while k < gamma and u_acc[k] < accept_prob(p_rows[k][drafts[k]], q_rows[k][drafts[k]]):
        k += 1
    if k < gamma:
        w = residual(p_rows[k], q_rows[k])
        if w is None:
            w, uu = p_rows[k], u_res
        else:
            uu = u_res
    else:
        w, uu = p_rows[gamma], u_bonus
    c = Fraction(0)
    tok = None
    for j, wj in enumerate(w):
        c += wj
        if c > uu:
            tok = j
            break
    if tok is None:
        tok = max(j for j, wj in enumerate(w) if wj > 0)
    return k, list(drafts[:k]) + [tok]
