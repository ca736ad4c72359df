"""Planted mistakes: each plausible slip in the fp64 oracle must make at least one pin fail.

A pin that no mistake can fail pins nothing. Here every mistake is applied to a copy of the oracle's
source text, loaded as a separate module on the CPU (the oracle itself is untouched), and a suite of
pins -- the pages' worked examples, the exact rational restatement, the reachable fp64 zero-residual
row, the strict accept test -- runs against the copy. The unmodified oracle must pass every pin; each
modified copy must fail at least one. CPU only.

The pins restate checks of tests/test_oracle.py in a form that takes the module under test as an
argument. Pages: [R] "Speculative decoding", rayaq.ca ml-models (Worked example; A round with a
rejection; One round, steps 3-5; The greedy case); [C] "Speculative decoding", cgnarendiran.github.io
blog (The correction that makes it exact).
"""
import importlib.util
import sys
from fractions import Fraction
from pathlib import Path

import numpy as np
import pytest

from conftest import load_golden
from oracle import exact
from test_oracle import _rand_simplex, logits_of, markov_round_inputs, zero_residual_row

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")   # log(0) = -inf logits

ORACLE_SRC = Path(__file__).resolve().parent.parent / "oracle" / "spec_verify_oracle.py"


def load_variant(name, old=None, new=None):
    """The oracle module built from its source with `old` replaced by `new` (exactly once)."""
    src = ORACLE_SRC.read_text()
    if old is not None:
        assert src.count(old) == 1, f"mutation site for {name!r} not unique: {old!r}"
        src = src.replace(old, new)
    modname = f"oracle_variant_{name}"
    spec = importlib.util.spec_from_loader(modname, loader=None)
    mod = importlib.util.module_from_spec(spec)
    sys.modules[modname] = mod          # dataclasses look their module up while the class is built
    try:
        exec(compile(src, f"<oracle variant {name}>", "exec"), mod.__dict__)
    finally:
        del sys.modules[modname]
    return mod


# ------------------------------------------------------------------------------------------------
# Pins, as functions of the module under test
# ------------------------------------------------------------------------------------------------

def _markov():
    g = load_golden("rayaq_markov_example.json")
    voc = g["vocabulary"]
    P = {voc.index(k): [Fraction(x) for x in v] for k, v in g["target_p"].items()}
    Q = {voc.index(k): [Fraction(x) for x in v] for k, v in g["draft_q"].items()}
    return g, voc, P, Q


def pin_rejection_round(m):
    """[R] A round with a rejection: ratios 1 and 5/7, u = 0.085 keeps, u = 0.835 rejects, the
    residual (1, 0, 0) forces 'a' for every residual uniform; emits 'c a'."""
    g, voc, P, Q = _markov()
    rr = g["rejection_round"]
    drafts = [voc.index(x) for x in rr["drafts"]]
    for u_res in (0.0, 0.3, 0.999):
        u = [rr["positions"][0]["u"], rr["positions"][1]["u"], 0.5, u_res, 0.5]
        r = m.oracle_verify(*markov_round_inputs(P, Q, voc.index("a"), drafts, u), diagnostics=True)
        row = r.rows[0]
        for i, pos in enumerate(rr["positions"]):
            assert abs(row.ratio[i] - float(Fraction(pos["ratio"]))) < 1e-12
        assert row.k == 1 and [voc[t] for t in row.tokens] == rr["emitted"]


def pin_alpha_per_context(m):
    """[R] Worked example: alpha 9/10, 4/5, 4/5 per context, through the batch outputs."""
    g, voc, P, Q = _markov()
    for name in voc:
        c = voc.index(name)
        zt = np.stack([logits_of(P[c]), logits_of(P[c])])[None]
        zd = logits_of(Q[c])[None, None]
        r = m.oracle_verify(zt, zd, np.array([[0]]), np.array([1]), np.ones(1, np.float32),
                            np.array([[0.5, 0.5, 0.5]], np.float32))
        assert abs(r.out_alpha[0, 0] - float(Fraction(g["alpha"][name]))) < 1e-12


def pin_four_token(m):
    """[C] The correction that makes it exact: ratio 0.5, alpha 0.70, residual (0, 2/3, 1/6, 1/6)."""
    g = load_golden("cgnarendiran_four_token.json")
    p = m.temperature_softmax(logits_of(g["target_p"]), 1.0)
    q = m.temperature_softmax(logits_of(g["draft_q"]), 1.0)
    x = g["tokens"].index(g["proposed"])
    assert abs(m.accept_ratio(p[x], q[x]) - g["accept_probability"]) < 1e-12
    w = m.residual_weights(p, q)
    np.testing.assert_allclose(w / w.sum(), [float(Fraction(s)) for s in g["residual_exact"]],
                               atol=1e-12)


def pin_exact_rule(m, trials=150):
    """Brute force against the exact rational restatement (oracle/exact.py, shared by no code):
    random tiny tables, rational uniforms, ragged draft lengths (the bonus row is gamma_b)."""
    rng = np.random.default_rng(21)
    checked = 0
    for _ in range(trials):
        V = int(rng.integers(2, 5))
        G = int(rng.integers(1, 4))
        gb = int(rng.integers(0, G + 1))
        den = 40
        P = [[Fraction(int(a), int(s)) for a, s in zip(*_rand_simplex(rng, V, den))]
             for _ in range(G + 1)]
        Q = [[Fraction(int(a), int(s)) for a, s in zip(*_rand_simplex(rng, V, den))] for _ in range(G)]
        drafts = [int(rng.choice(V, p=[float(v) for v in Q[i]])) for i in range(G)]
        u = [Fraction(int(rng.integers(0, 997)), 997) for _ in range(G + 2)]
        k_ex, toks_ex = exact.verify_row_exact(P[:gb + 1], Q[:gb], drafts[:gb], u[:gb], u[G],
                                               u[G + 1])
        zt = np.stack([logits_of(p) for p in P])[None]
        zd = np.stack([logits_of(q) for q in Q])[None]
        r = m.oracle_verify(zt, zd, np.asarray([drafts], np.int32), np.asarray([gb]),
                            np.ones(1, np.float32), np.asarray([[float(x) for x in u]], np.float64),
                            diagnostics=True, eps=1e-9)
        if not r.rows[0].exact:
            continue
        checked += 1
        assert r.rows[0].k == k_ex and r.rows[0].tokens == toks_ex
    assert checked > trials // 2


def pin_zero_residual_fallback(m):
    """The fp64 row whose residual rounds to zero mass: the draw comes from p with u[G]."""
    zt, zd, x = zero_residual_row(64)
    p = m.temperature_softmax(zt[0], 1.0)
    u = np.array([0.9, 0.05, 0.81], np.float32)
    res = m.verify_row(zt, zd, np.asarray([x]), 1, np.float32(1.0), u, 1)
    assert res.k == 0
    c = np.cumsum(p)
    assert res.tokens == [int(np.flatnonzero(c > np.float64(u[1]) * c[-1])[0])]


def pin_strict_accept(m):
    """[R] One round, step 3: keep x only while u < min(1, p/q); u equal to the ratio 1/2 rejects."""
    zt = np.zeros((1, 2, 2))
    zd = np.array([[[0.0, -np.inf]]])
    for u0, k in ((0.5, 0), (np.nextafter(np.float32(0.5), np.float32(0)), 1)):
        u = np.array([[u0, 0.25, 0.25]], np.float32)
        r = m.oracle_verify(zt, zd, np.array([[0]]), np.array([1]), np.ones(1, np.float32), u)
        assert r.out_num_emitted[0] - 1 == k


def pin_zero_mass_token(m):
    """A drafted token that both p and q give zero mass is rejected ([R] The output distribution is
    exactly the target's), while q(x) = 0 with p(x) > 0 keeps it."""
    zt = np.log(np.array([[[0.5, 0.5, 0.0], [0.2, 0.3, 0.5]]]))
    for zx_d, k in ((-np.inf, 0), (0.0, None)):
        zd = np.array([[[0.0, 0.0, zx_d]]]) if zx_d == 0.0 else np.log(np.array([[[0.5, 0.5, 0.0]]]))
        r = m.oracle_verify(zt, zd, np.array([[2]]), np.array([1]), np.ones(1, np.float32),
                            np.array([[0.99, 0.5, 0.5]], np.float32))
        if k is not None:
            assert r.out_num_emitted[0] - 1 == k and r.out_tokens[0, 0] != 2
    zd = np.log(np.array([[[0.5, 0.5, 0.0]]]))
    zt2 = np.log(np.array([[[0.4, 0.4, 0.2], [0.2, 0.3, 0.5]]]))
    r = m.oracle_verify(zt2, zd, np.array([[2]]), np.array([1]), np.ones(1, np.float32),
                        np.array([[0.99, 0.5, 0.5]], np.float32))
    assert r.out_num_emitted[0] == 2 and r.out_tokens[0, 0] == 2


def pin_strict_draw(m):
    """The draw's inverse CDF takes the first token whose running weight is strictly above u times
    the total: p = (0, 1/2, 1/2) on the bonus row gives token 1 for u = 0 (a zero-weight token is
    never chosen) and token 2 for u = 1/2 (a threshold on a boundary goes to the next token)."""
    zt = np.log(np.array([[[0.0, 0.5, 0.5]]]))
    for ub, want in ((0.0, 1), (0.5, 2)):
        r = m.oracle_verify(zt, np.zeros((1, 0, 3)), np.zeros((1, 0), np.int32), np.array([0]),
                            np.ones(1, np.float32), np.array([[0.5, ub]], np.float32))
        assert list(r.out_tokens[0]) == [want]


def pin_greedy_ties(m):
    """Greedy: argmax ties go to the lowest index ([R] The greedy case)."""
    zt = np.zeros((1, 2, 6))
    zt[0, 0, [2, 4]] = 5.0
    zt[0, 1, [1, 3]] = 1.0
    r = m.oracle_verify(zt, None, np.asarray([[2]]), np.asarray([1]), np.zeros(1, np.float32),
                        np.zeros((1, 3), np.float32))
    assert list(r.out_tokens[0]) == [2, 1] and r.out_num_emitted[0] == 2


def pin_equal_rows_any_temperature(m):
    """p = q at every position (the same logits, one temperature for both) accepts every draft."""
    rng = np.random.default_rng(8)
    V, G = 50, 6
    z = rng.normal(0, 2, (1, G + 1, V))
    x = rng.integers(0, V, (1, G)).astype(np.int32)
    u = rng.random((1, G + 2)).astype(np.float32)
    r = m.oracle_verify(z, z[:, :G], x, np.asarray([G]), np.full(1, 0.6, np.float32), u)
    assert r.out_num_emitted[0] == G + 1
    np.testing.assert_allclose(r.out_alpha[0], 1.0, atol=1e-12)


PINS = [pin_rejection_round, pin_alpha_per_context, pin_four_token, pin_exact_rule,
        pin_zero_residual_fallback, pin_strict_accept, pin_zero_mass_token, pin_strict_draw,
        pin_greedy_ties,
        pin_equal_rows_any_temperature]

# (name, text in the oracle, replacement): the slips the pins must catch.
MISTAKES = [
    ("swapped ratio", "return min(1.0, p_x / q_x)", "return min(1.0, q_x / p_x)"),
    ("<= in the accept test", "np.float64(u[k]) < ratio[k]:", "np.float64(u[k]) <= ratio[k]:"),
    (">= in the CDF", "hit = np.flatnonzero(c > t)", "hit = np.flatnonzero(c >= t)"),
    ("flipped residual sign", "np.maximum(0.0, p - q)", "np.maximum(0.0, q - p)"),
    ("residual of the wrong position", "w = residual_weights(p_rows[kk], q_rows[kk])",
     "w = residual_weights(p_rows[gamma_b - 1], q_rows[gamma_b - 1])"),
    ("bonus uniform for the residual", "            uu = np.float64(u[G])\n",
     "            uu = np.float64(u[G + 1])\n"),
    ("residual uniform for the bonus", "            uu = np.float64(u[G + 1])\n",
     "            uu = np.float64(u[G])\n"),
    ("bonus from row G", "p_bonus = dist(zt[gamma_b])", "p_bonus = dist(zt[G])"),
    ("fallback with the bonus uniform", "                w = p_rows[kk]\n",
     "                w = p_rows[kk]\n                uu = np.float64(u[G + 1])\n"),
    ("fallback to the last token", "                w = p_rows[kk]\n",
     "                w = np.eye(len(p_rows[kk]))[-1]\n"),
    ("alpha as sum max(p, q)", "alpha[i] = np.sum(np.minimum(p, q))",
     "alpha[i] = np.sum(np.maximum(p, q))"),
    ("zero-mass token kept", "return 1.0 if p_x > 0.0 else 0.0", "return 1.0"),
    ("greedy ties to the highest index", "return int(np.argmax(np.asarray(z, dtype=np.float64)))",
     "return int(len(z) - 1 - np.argmax(np.asarray(z, dtype=np.float64)[::-1]))"),
    ("temperature on p only", "        q = dist(zd[i])\n",
     "        q = filtered_softmax(zd[i], 1.0, top_k, top_p)[0]\n"),
]


def failing_pins(m):
    failed = []
    for pin in PINS:
        try:
            pin(m)
        except Exception as e:            # an assertion, or a crash the slip causes
            failed.append((pin.__name__, type(e).__name__))
    return failed


def test_unmodified_oracle_passes_every_pin():
    assert failing_pins(load_variant("unmodified")) == []


@pytest.mark.parametrize("name,old,new", MISTAKES, ids=[m[0] for m in MISTAKES])
def test_planted_mistake_fails_a_pin(name, old, new):
    failed = failing_pins(load_variant(name.replace(" ", "_"), old, new))
    assert failed, f"no pin catches the planted mistake {name!r}"
