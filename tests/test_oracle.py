"""Pins of the fp64 oracle to facts the pages fix: printed worked examples, closed forms, identities,
special cases and an exact rational-arithmetic restatement on tiny inputs. CPU only."""
from fractions import Fraction

import numpy as np
import pytest

from conftest import load_golden
from oracle import exact
from oracle.spec_verify_oracle import (accept_ratio, admissible_draws, inverse_cdf, oracle_verify,
                                       residual_weights, sample_drafts, temperature_softmax,
                                       verify_row)


def logits_of(p):
    """Logits whose T=1 softmax is p (log p; -inf where p = 0)."""
    p = np.asarray([float(x) for x in p], dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.log(p)


def markov_round_inputs(P, Q, start, drafts, u):
    """Target rows p(.|ctx_i) for i = 0..gamma (ctx_0 = start, ctx_i = draft i-1) and draft rows
    q(.|ctx_i) for i < gamma, as logits, in the oracle's [1, G+1, V] / [1, G, V] layout."""
    ctx = [start] + list(drafts)
    zt = np.stack([logits_of(P[c]) for c in ctx])[None]
    zd = np.stack([logits_of(Q[c]) for c in ctx[:-1]])[None]
    G = len(drafts)
    return zt, zd, np.asarray([drafts], np.int32), np.asarray([G], np.int32), \
        np.ones(1, np.float32), np.asarray([u], np.float32)


# -------------------------------------------------------------------------------------------------
# rayaq.ca worked example
# -------------------------------------------------------------------------------------------------

def test_markov_alpha_and_residual_exact(markov):
    g, voc, P, Q = markov
    for name in voc:
        c = voc.index(name)
        assert exact.alpha(P[c], Q[c]) == Fraction(g["alpha"][name])
        assert exact.residual(P[c], Q[c]) == [Fraction(x) for x in g["residual"][name]]


def test_markov_alpha_and_residual_float_oracle(markov):
    g, voc, P, Q = markov
    for name in voc:
        c = voc.index(name)
        p = temperature_softmax(logits_of(P[c]), 1.0)
        q = temperature_softmax(logits_of(Q[c]), 1.0)
        assert np.sum(np.minimum(p, q)) == pytest.approx(float(Fraction(g["alpha"][name])), abs=1e-12)
        w = residual_weights(p, q)
        want = [float(Fraction(x)) for x in g["residual"][name]]
        np.testing.assert_allclose(w / w.sum(), want, atol=1e-12)


def test_rejection_round(markov):
    g, voc, P, Q = markov
    rr = g["rejection_round"]
    a = voc.index("a")
    drafts = [voc.index(x) for x in rr["drafts"]]
    for u_res in (0.0, 0.3, 0.999):
        u = [rr["positions"][0]["u"], rr["positions"][1]["u"], 0.5, u_res, 0.5]
        r = oracle_verify(*markov_round_inputs(P, Q, a, drafts, u), diagnostics=True)
        row = r.rows[0]
        for i, pos in enumerate(rr["positions"]):
            assert row.ratio[i] == pytest.approx(float(Fraction(pos["ratio"])), abs=1e-12)
            assert r.out_p_draft[0, i] == pytest.approx(float(Fraction(pos["p"])), abs=1e-12)
            assert r.out_q_draft[0, i] == pytest.approx(float(Fraction(pos["q"])), abs=1e-12)
        assert row.k == 1
        assert [voc[t] for t in row.tokens] == rr["emitted"]
        assert r.out_num_emitted[0] == 2
        assert list(r.out_tokens[0]) == [voc.index("c"), voc.index("a"), -1, -1]


def test_all_accept_round(markov):
    """The page's seed-0 round: b, c, c all pass and a bonus 'c' follows. The uniforms are not
    printed, so they are placed below each exact ratio (3/4, 1, 5/7) and the bonus uniform in the
    'c' interval of p(.|c) = (3/10, 1/5, 1/2)."""
    g, voc, P, Q = markov
    ar = g["all_accept_round"]
    drafts = [voc.index(x) for x in ar["drafts"]]
    u = [0.74, 0.99, 0.71, 0.9, 0.6]
    r = oracle_verify(*markov_round_inputs(P, Q, voc.index("a"), drafts, u), diagnostics=True)
    assert [voc[t] for t in r.rows[0].tokens] == ar["emitted"]
    np.testing.assert_allclose(r.rows[0].ratio, [0.75, 1.0, 5 / 7], atol=1e-12)
    assert r.rows[0].exact


def test_round_enumeration_and_accept_distribution(markov):
    g, voc, P, Q = markov
    seqs, pk = exact.round_outcomes(lambda c: P[c], lambda c: Q[c], voc.index("a"), 3)
    assert len(seqs) == g["distinct_sequences_one_round"]
    assert sum(seqs.values()) == 1
    assert pk == [Fraction(x) for x in g["accept_count_distribution"]]
    mean = sum((k + 1) * p for k, p in enumerate(pk))
    assert mean == Fraction(g["mean_tokens_per_round"])
    assert round(float(mean), 2) == g["mean_tokens_per_round_decimal"]
    a0 = float(exact.alpha(P[0], Q[0]))
    assert round((1 - a0 ** 4) / (1 - a0), 3) == g["iid_formula_prediction"]


def test_two_token_joint_equals_target(markov):
    g, voc, P, Q = markov
    joint = exact.joint_first_tokens(lambda c: P[c], lambda c: Q[c], voc.index("a"), 3, 2)
    for key, val in g["two_token_joint"].items():
        t = tuple(voc.index(ch) for ch in key)
        assert joint[t] == Fraction(val)
        assert joint[t] == P[voc.index("a")][t[0]] * P[t[0]][t[1]]


def test_three_token_joint_every_context(markov):
    """Exactness from every starting context, three tokens deep (the page's tests check the same)."""
    g, voc, P, Q = markov
    for start in range(3):
        joint = exact.joint_first_tokens(lambda c: P[c], lambda c: Q[c], start, 2, 3)
        for t, val in joint.items():
            assert val == P[start][t[0]] * P[t[0]][t[1]] * P[t[1]][t[2]]
        assert sum(joint.values()) == 1


# -------------------------------------------------------------------------------------------------
# cgnarendiran.github.io four-token example and quiz values
# -------------------------------------------------------------------------------------------------

def test_four_token_example():
    g = load_golden("cgnarendiran_four_token.json")
    p = temperature_softmax(logits_of(g["target_p"]), 1.0)
    q = temperature_softmax(logits_of(g["draft_q"]), 1.0)
    x = g["tokens"].index(g["proposed"])
    assert accept_ratio(p[x], q[x]) == pytest.approx(g["accept_probability"], abs=1e-12)
    alpha = np.sum(np.minimum(p, q))
    assert alpha == pytest.approx(g["alpha"], abs=1e-12)
    assert 1 - alpha == pytest.approx(g["rejection_probability"], abs=1e-12)
    w = residual_weights(p, q)
    np.testing.assert_allclose(w / w.sum(), [float(Fraction(s)) for s in g["residual_exact"]],
                               atol=1e-12)
    np.testing.assert_allclose(w / w.sum(), g["residual"], atol=5e-4)
    # emit probabilities, exactly: P(emit y) = sum_x q(x) [a(x) 1{y=x} + (1 - a(x)) r(y)]
    P = [Fraction(s).limit_denominator(100) for s in map(str, g["target_p"])]
    Q = [Fraction(s).limit_denominator(100) for s in map(str, g["draft_q"])]
    r = exact.residual(P, Q)
    emit = [sum(Q[xx] * (exact.accept_prob(P[xx], Q[xx]) * (y == xx)
                         + (1 - exact.accept_prob(P[xx], Q[xx])) * r[y]) for xx in range(4))
            for y in range(4)]
    assert emit == P
    for name, val in g["emit_probability"].items():
        assert float(emit[g["tokens"].index(name)]) == pytest.approx(val, abs=1e-12)


def test_quiz_ratio_and_kept_when_p_ge_q():
    g = load_golden("formula_values.json")
    for item in g["accept_ratio"]:
        assert accept_ratio(item["p"], item["q"]) == pytest.approx(item["value"], abs=1e-15)
    assert accept_ratio(0.5, 0.2) == 1.0
    assert accept_ratio(0.3, 0.3) == 1.0
    # q(x) = 0 reading: kept when the target gives x mass, rejected when it gives none (a token of
    # zero target mass is never emitted: [R] The output distribution is exactly the target's)
    assert accept_ratio(0.25, 0.0) == 1.0
    assert accept_ratio(0.0, 0.0) == 0.0


def test_expected_tokens_closed_form_matches_pages():
    g = load_golden("formula_values.json")
    for item in g["expected_tokens_per_round"]:
        a, gam = item["alpha"], item["gamma"]
        assert round((1 - a ** (gam + 1)) / (1 - a), item["decimals"]) == item["value"]


# -------------------------------------------------------------------------------------------------
# Identities and special cases
# -------------------------------------------------------------------------------------------------

def test_identities_random_rows():
    rng = np.random.default_rng(11)
    for V in (2, 5, 64, 1000):
        for _ in range(20):
            zt = rng.normal(0, 2, V)
            zd = zt + rng.normal(0, rng.uniform(0.1, 3), V)
            T = rng.uniform(0.3, 2.0)
            p, q = temperature_softmax(zt, T), temperature_softmax(zd, T)
            w = residual_weights(p, q)
            alpha = np.sum(np.minimum(p, q))
            np.testing.assert_allclose(np.minimum(p, q) + w, p, atol=1e-15)
            assert np.sum(w) == pytest.approx(1 - alpha, abs=1e-12)
            assert alpha == pytest.approx(1 - 0.5 * np.sum(np.abs(p - q)), abs=1e-12)
            assert np.sum(p) == pytest.approx(1.0, abs=1e-12)


def test_softmax_special_cases():
    V = 37
    np.testing.assert_allclose(temperature_softmax(np.full(V, 3.25), 0.7), np.full(V, 1 / V),
                               rtol=1e-14)
    rng = np.random.default_rng(3)
    p = rng.dirichlet(np.ones(V))
    np.testing.assert_allclose(temperature_softmax(np.log(p), 1.0), p, rtol=1e-12)
    # temperature T on logits z equals T = 1 on z / T; a constant shift changes nothing
    z = rng.normal(0, 3, V)
    np.testing.assert_allclose(temperature_softmax(z, 0.5), temperature_softmax(2 * z, 1.0),
                               rtol=1e-12)
    np.testing.assert_allclose(temperature_softmax(z + 1e3, 1.0), temperature_softmax(z, 1.0),
                               rtol=1e-10)
    # -inf logits carry no mass
    z[5] = -np.inf
    assert temperature_softmax(z, 1.0)[5] == 0.0


def test_inverse_cdf_rules():
    w = np.array([0.0, 0.25, 0.0, 0.5, 0.25])
    assert inverse_cdf(w, 0.0) == 1            # strict '>' skips the zero-weight head
    assert inverse_cdf(w, 0.2499) == 1
    assert inverse_cdf(w, 0.25) == 3           # C = 0.25 is not > 0.25: next positive token
    assert inverse_cdf(w, 0.7499) == 3
    assert inverse_cdf(w, 0.75) == 4
    assert inverse_cdf(w, 0.999999) == 4
    assert inverse_cdf(w, 1.0) == 4            # overrun: last positive token
    for u in np.linspace(0, 0.999, 200):
        assert w[inverse_cdf(w, u)] > 0
    # frequencies over a fine grid of u equal the weights (the draw is a sample of w / sum w)
    us = (np.arange(100000) + 0.5) / 100000
    counts = np.bincount([inverse_cdf(w, u) for u in us[::10]], minlength=5) / len(us[::10])
    np.testing.assert_allclose(counts, w, atol=2e-4)


def test_admissible_draws_margin():
    w = np.array([0.25, 0.25, 0.5])
    toks, gap = admissible_draws(w, 0.5, 1e-5)        # threshold exactly on a boundary
    assert toks == [1, 2] and gap == pytest.approx(0.0)
    toks, gap = admissible_draws(w, 0.6, 1e-5)
    assert toks == [2] and gap == pytest.approx(0.1)


def test_greedy_equals_plain_greedy_decoding():
    """Greedy verification over arbitrary drafts reproduces plain greedy decoding of the target
    token for token (rayaq.ca, The greedy case; brunomaga.github.io, greedy rule)."""
    rng = np.random.default_rng(5)
    V, G, n_out = 11, 4, 40
    table = rng.normal(0, 2, (V, V))             # target logits after token c: table[c]
    plain = [0]
    while len(plain) < n_out + 1:
        plain.append(int(np.argmax(table[plain[-1]])))
    seq = [0]
    while len(seq) < n_out + 1:
        drafts = [int(np.argmax(table[seq[-1]])) if rng.random() < 0.6 else int(rng.integers(V))]
        for _ in range(G - 1):
            drafts.append(int(np.argmax(table[drafts[-1]])) if rng.random() < 0.7
                          else int(rng.integers(V)))
        ctx = [seq[-1]] + drafts
        zt = np.stack([table[c] for c in ctx])[None]
        r = oracle_verify(zt, np.zeros((1, G, V)), np.asarray([drafts]), np.asarray([G]),
                          np.zeros(1, np.float32), np.zeros((1, G + 2), np.float32))
        n = r.out_num_emitted[0]
        assert 1 <= n <= G + 1
        seq.extend(int(t) for t in r.out_tokens[0, :n])
        assert r.out_alpha[0, :n - 1].tolist() == [1.0] * (n - 1)
    assert seq[:n_out + 1] == plain[:n_out + 1]


def test_greedy_argmax_ties_lowest_index():
    zt = np.zeros((1, 2, 6))
    zt[0, 0, [2, 4]] = 5.0
    zt[0, 1, [1, 3]] = 1.0
    r = oracle_verify(zt, None, np.asarray([[2]]), np.asarray([1]), np.zeros(1, np.float32),
                      np.zeros((1, 3), np.float32))
    assert list(r.out_tokens[0]) == [2, 1] and r.out_num_emitted[0] == 2


def test_equal_distributions_accept_everything():
    rng = np.random.default_rng(8)
    V, G = 50, 6
    z = rng.normal(0, 2, (1, G + 1, V))
    x = rng.integers(0, V, (1, G)).astype(np.int32)
    u = rng.random((1, G + 2)).astype(np.float32)
    r = oracle_verify(z, z[:, :G], x, np.asarray([G]), np.ones(1, np.float32), u)
    assert r.out_num_emitted[0] == G + 1
    np.testing.assert_allclose(r.out_alpha[0], 1.0, atol=1e-12)
    # greedy with drafts equal to the argmax: all accepted plus the bonus argmax
    xg = np.argmax(z[0, :G], axis=-1)[None].astype(np.int32)
    r = oracle_verify(z, None, xg, np.asarray([G]), np.zeros(1, np.float32), u)
    assert r.out_num_emitted[0] == G + 1 and r.out_tokens[0, G] == np.argmax(z[0, G])


def test_float_oracle_matches_exact_rule_on_tiny_inputs():
    """Brute force against the exact restatement: random tiny tables, random rational uniforms.
    Cases within 1e-9 of a decision boundary are skipped (rounding may legitimately differ)."""
    rng = np.random.default_rng(21)
    checked = skipped = 0
    for trial in range(400):
        V = int(rng.integers(2, 5))
        G = int(rng.integers(0, 4))
        den = 40
        P = [[Fraction(int(a), int(s)) for a, s in zip(*_rand_simplex(rng, V, den))] for _ in range(G + 1)]
        Q = [[Fraction(int(a), int(s)) for a, s in zip(*_rand_simplex(rng, V, den))] for _ in range(G)]
        drafts = [int(rng.choice(V, p=[float(v) for v in Q[i]])) for i in range(G)]
        u = [Fraction(int(rng.integers(0, 997)), 997) for _ in range(G + 2)]
        k_ex, toks_ex = exact.verify_row_exact(P, Q, drafts, u[:G], u[G], u[G + 1])
        zt = np.stack([logits_of(p) for p in P])[None]
        zd = np.stack([logits_of(q) for q in Q])[None] if G else np.zeros((1, 0, V))
        r = oracle_verify(zt, zd, np.asarray([drafts], np.int32).reshape(1, G), np.asarray([G]),
                          np.ones(1, np.float32), np.asarray([[float(x) for x in u]], np.float64),
                          diagnostics=True, eps=1e-9)
        if not r.rows[0].exact:
            skipped += 1
            continue
        checked += 1
        assert r.rows[0].k == k_ex and r.rows[0].tokens == toks_ex, (trial, P, Q, drafts, u)
    assert checked > 300 and skipped < 60


def _rand_simplex(rng, V, den):
    cuts = np.sort(rng.integers(0, den + 1, V - 1))
    parts = np.diff(np.concatenate(([0], cuts, [den])))
    return parts, [den] * V


def test_sample_drafts_distribution():
    rng = np.random.default_rng(4)
    q_logits = np.log(np.array([[[0.6, 0.2, 0.15, 0.05]]]))
    u = rng.random((1, 1)).astype(np.float32)
    assert sample_drafts(q_logits, np.ones(1, np.float32), u)[0, 0] in range(4)
    us = (np.arange(4000) + 0.5) / 4000
    xs = [sample_drafts(q_logits, np.ones(1, np.float32), np.asarray([[v]]))[0, 0] for v in us]
    np.testing.assert_allclose(np.bincount(xs, minlength=4) / 4000, [0.6, 0.2, 0.15, 0.05], atol=1e-3)


# -------------------------------------------------------------------------------------------------
# Row-error rules
# -------------------------------------------------------------------------------------------------

def _small_row(G=3, V=8, T=1.0, seed=0):
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, 1, (1, G + 1, V))
    zd = rng.normal(0, 1, (1, G, V))
    x = rng.integers(0, V, (1, G)).astype(np.int32)
    u = rng.random((1, G + 2)).astype(np.float32)
    return zt, zd, x, np.asarray([G], np.int32), np.asarray([T], np.float32), u


@pytest.mark.parametrize("case", ["len_neg", "len_big", "T_nan", "T_neg", "T_inf", "T_subnormal",
                                  "tok_neg", "tok_big", "u_one", "u_nan", "nan_logit",
                                  "pinf_logit", "all_ninf", "draft_nan"])
def test_row_errors(case):
    zt, zd, x, n, T, u = _small_row()
    if case == "len_neg":
        n[0] = -1
    elif case == "len_big":
        n[0] = 4
    elif case == "T_nan":
        T[0] = np.nan
    elif case == "T_neg":
        T[0] = -0.5
    elif case == "T_inf":
        T[0] = np.inf
    elif case == "T_subnormal":
        T[0] = np.float32(1e-40)
    elif case == "tok_neg":
        x[0, 1] = -1
    elif case == "tok_big":
        x[0, 2] = 8
    elif case == "u_one":
        u[0, 3] = 1.0
    elif case == "u_nan":
        u[0, 0] = np.nan
    elif case == "nan_logit":
        zt[0, 3, 2] = np.nan
    elif case == "pinf_logit":
        zt[0, 1, 0] = np.inf
    elif case == "all_ninf":
        zt[0, 0, :] = -np.inf
    elif case == "draft_nan":
        zd[0, 2, 7] = np.nan
    r = oracle_verify(zt, zd, x, n, T, u)
    assert r.out_num_emitted[0] == -1
    assert (r.out_tokens[0] == -1).all()
    assert (r.out_alpha[0] == 0).all()


def test_padding_and_greedy_ignore_unused_inputs():
    zt, zd, x, n, T, u = _small_row(G=4)
    n[0] = 2
    zt[0, 3:] = np.nan         # target rows past gamma_b
    zd[0, 2:] = np.nan         # draft rows at or past gamma_b
    x[0, 2:] = -1
    u[0, 2:4] = np.nan          # accept uniforms past gamma_b (column G and G+1 are used)
    u[0, 4:] = 0.5
    r = oracle_verify(zt, zd, x, n, T, u)
    assert r.out_num_emitted[0] >= 1
    assert (r.out_alpha[0, 2:] == 0).all()
    # greedy rows read neither draft logits nor uniforms
    zt, zd, x, n, T, u = _small_row(G=3)
    zd[:] = np.nan
    u[:] = np.nan
    T[0] = 0.0
    r = oracle_verify(zt, zd, x, n, T, u)
    assert r.out_num_emitted[0] >= 1


def test_zero_draft_length():
    zt, zd, x, n, T, u = _small_row(G=3)
    n[0] = 0
    r = oracle_verify(zt, zd, x, n, T, u)
    assert r.out_num_emitted[0] == 1
    p = temperature_softmax(zt[0, 0], 1.0)
    assert r.out_tokens[0, 0] == inverse_cdf(p, np.float64(u[0, 4]))


def zero_residual_row(V, x=3, seed=3, dtype=np.float32):
    """One drafted position whose fp64 residual max(0, p - q) has zero total mass although
    p(x) < q(x): every logit but x's is the same in both rows, and x's logit (-40 in the target, -39
    in the draft) is so small that its term vanishes in both normalisers. So p and q agree exactly
    everywhere but at x, where p(x)/q(x) = e^-1. (In exact arithmetic the residual is p without x,
    whose draw matches the fallback's draw from p.) Returns (zt [2, V], zd [1, V], x)."""
    rng = np.random.default_rng(seed)
    base = np.abs(rng.standard_normal(V)).astype(dtype)
    zt, zd = base.copy(), base.copy()
    zt[x], zd[x] = -40.0, -39.0
    return np.stack([zt, base]), zd[None], x


@pytest.mark.parametrize("V", [8, 64, 4096])
def test_verify_row_residual_fallback_zero_mass(V):
    """A rejection whose residual has zero mass draws from that position's p with the residual
    uniform u[G] (the reading for a step the pages leave open: [R] One round, step 4 cannot divide
    by a zero mass). The case is a real one: fp64 rounding leaves the residual exactly empty."""
    zt, zd, x = zero_residual_row(V)
    p = temperature_softmax(zt[0], 1.0)
    q = temperature_softmax(zd[0], 1.0)
    assert np.sum(residual_weights(p, q)) == 0.0          # the fallback's condition, reached
    assert p[x] < q[x]
    assert accept_ratio(p[x], q[x]) == pytest.approx(np.exp(-1.0), rel=1e-12)
    u = np.array([0.9, 0.05, 0.81], np.float32)          # u[0] rejects; u[G] = 0.05; u[G+1] = 0.81
    res = verify_row(zt, zd, np.asarray([x]), 1, np.float32(1.0), u, 1, diagnostics=True)
    assert res.k == 0
    want = inverse_cdf(p, np.float64(u[1]))
    assert res.tokens == [want]
    # the mistakes this branch could hide give other tokens on this row
    assert want != inverse_cdf(p, np.float64(u[2]))                 # the bonus uniform
    assert want != int(np.flatnonzero(p > 0)[-1])                   # the last token
    assert want != int(np.argmax(p))                                 # the mode
    assert want != x                                                  # the rejected draft
    assert res.exact


def test_accept_is_strict_at_the_ratio():
    """Keep x only when u < min(1, p/q) (rayaq.ca, One round, step 3): u equal to the ratio rejects.
    p = (1/2, 1/2) and q = (1, 0) give the exactly representable ratio 1/2 for x = 0."""
    zt = np.zeros((1, 2, 2))
    zd = np.array([[[0.0, -np.inf]]])
    for u0, k in ((0.5, 0), (np.nextafter(np.float32(0.5), np.float32(0)), 1)):
        u = np.array([[u0, 0.25, 0.25]], np.float32)
        r = oracle_verify(zt, zd, np.array([[0]]), np.array([1]), np.ones(1, np.float32), u)
        assert r.out_num_emitted[0] - 1 == k


def test_threaded_row_driver_equals_the_batch_oracle():
    """oracle_verify_rows (rows in a thread pool) gives what oracle_verify gives, row for row."""
    from oracle.spec_verify_oracle import oracle_verify_rows
    zt, zd, x, n, T, u = _small_row(G=3, V=40, seed=11)
    rng = np.random.default_rng(12)
    B = 9
    zt = np.concatenate([zt] * B) + rng.normal(0, 1, (B,) + zt.shape[1:])
    zd = np.concatenate([zd] * B) + rng.normal(0, 1, (B,) + zd.shape[1:])
    x = np.concatenate([x] * B)
    n = rng.integers(0, 4, B).astype(np.int32)
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    T[2] = 0.0
    u = rng.random((B, 5), dtype=np.float32)
    ref = oracle_verify(zt, zd, x, n, T, u, diagnostics=True)
    rows = [0, 2, 3, 5, 8]
    got = oracle_verify_rows(lambda b: (zt[b], zd[b]), x, n, T, u, 3, 40, rows, threads=3,
                             diagnostics=True)
    for b in range(B):
        if b in rows:
            assert got.rows[b].tokens == ref.rows[b].tokens and got.rows[b].k == ref.rows[b].k
            assert np.array_equal(got.out_alpha[b], ref.out_alpha[b])
            assert got.rows[b].exact == ref.rows[b].exact
        else:
            assert got.rows[b] is None and got.out_num_emitted[b] == -1
    assert np.array_equal(got.out_tokens[rows], ref.out_tokens[rows])
