"""Monte-Carlo pins of the fp64 oracle: with drafts sampled from q and fresh uniforms, the emitted
token is distributed as the target p, the accept count follows the pages' exact distribution, and
the mean tokens per round under identical positions equals (1 - a^(g+1)) / (1 - a). CPU only,
fixed seeds (deterministic)."""
from fractions import Fraction

import numpy as np
import pytest
from scipy import stats

from conftest import load_golden
from oracle.spec_verify_oracle import oracle_verify


def _sample(rng, dist, n):
    return rng.choice(len(dist), size=n, p=np.asarray(dist, dtype=np.float64))


def test_emitted_token_distributed_as_target():
    """cgnarendiran.github.io four-token example: one drafted position, draft ~ q; the first emitted
    token must follow p (chi-square, fixed seed)."""
    g = load_golden("cgnarendiran_four_token.json")
    p, q = np.array(g["target_p"]), np.array(g["draft_q"])
    rng = np.random.default_rng(1234)
    N = 20000
    x = _sample(rng, q, N).astype(np.int32)[:, None]
    zt = np.broadcast_to(np.log(np.stack([p, p])), (N, 2, 4))
    zd = np.broadcast_to(np.log(q)[None], (N, 1, 4))
    u = rng.random((N, 3)).astype(np.float32)
    r = oracle_verify(zt, zd, x, np.ones(N, np.int32), np.ones(N, np.float32), u)
    first = r.out_tokens[:, 0]
    counts = np.bincount(first, minlength=4)
    chi = stats.chisquare(counts, N * p)
    assert chi.pvalue > 1e-3, (counts, N * p)
    # acceptance rate equals alpha = 0.7
    acc = np.mean(r.out_num_emitted == 2)
    assert abs(acc - g["alpha"]) < 4 * np.sqrt(0.21 / N)


@pytest.mark.parametrize("item", load_golden("formula_values.json")["expected_tokens_per_round"])
def test_mean_tokens_per_round_iid(item):
    """Identical (p, q) at every position with sum min(p, q) = alpha: the mean of k + 1 equals the
    closed form the pages print (within 4 standard errors)."""
    a, G = item["alpha"], item["gamma"]
    if a == 0.8:
        p, q = np.array([0.9, 0.1]), np.array([0.7, 0.3])
    else:
        p, q = np.array([0.15, 0.85]), np.array([0.85, 0.15])
    assert np.sum(np.minimum(p, q)) == pytest.approx(a)
    rng = np.random.default_rng(99 + G)
    N = 12000
    x = _sample(rng, q, N * G).astype(np.int32).reshape(N, G)
    zt = np.broadcast_to(np.log(p), (N, G + 1, 2))
    zd = np.broadcast_to(np.log(q), (N, G, 2))
    u = rng.random((N, G + 2)).astype(np.float32)
    r = oracle_verify(zt, zd, x, np.full(N, G, np.int32), np.ones(N, np.float32), u)
    n = r.out_num_emitted.astype(np.float64)
    closed = (1 - a ** (G + 1)) / (1 - a)
    assert round(closed, item["decimals"]) == item["value"]
    assert abs(n.mean() - closed) < 4 * n.std() / np.sqrt(N), (n.mean(), closed)


def test_accept_count_distribution_markov_round(markov):
    """rayaq.ca round from 'a' with gamma = 3: drafts drawn from the Markov draft model, verified
    against the matching target rows; the accept-count histogram follows 1/10, 13/100, 61/500,
    81/125 (chi-square, fixed seed), and the emitted first token follows p(. | a)."""
    g, voc, P, Q = markov
    Pf = {c: np.array([float(v) for v in P[c]]) for c in P}
    Qf = {c: np.array([float(v) for v in Q[c]]) for c in Q}
    rng = np.random.default_rng(77)
    N, G = 12000, 3
    zt = np.empty((N, G + 1, 3))
    zd = np.empty((N, G, 3))
    x = np.empty((N, G), np.int32)
    for n in range(N):
        ctx = voc.index("a")
        for i in range(G):
            zt[n, i] = np.log(Pf[ctx])
            zd[n, i] = np.log(Qf[ctx])
            x[n, i] = rng.choice(3, p=Qf[ctx])
            ctx = x[n, i]
        zt[n, G] = np.log(Pf[ctx])
    u = rng.random((N, G + 2)).astype(np.float32)
    r = oracle_verify(zt, zd, x, np.full(N, G, np.int32), np.ones(N, np.float32), u)
    k = r.out_num_emitted - 1
    want = np.array([float(Fraction(s)) for s in g["accept_count_distribution"]])
    chi = stats.chisquare(np.bincount(k, minlength=4), N * want)
    assert chi.pvalue > 1e-3
    first = np.bincount(r.out_tokens[:, 0], minlength=3)
    chi = stats.chisquare(first, N * Pf[voc.index("a")])
    assert chi.pvalue > 1e-3
