"""Top-k / top-p filtering before the test: oracle pins on the CPU and GPU parity of
spec_verify_filtered.

[R] "Speculative decoding" (rayaq.ca), Why the output is exactly the target's: temperature, top-p
and any penalties are applied to p and q before the test, because the rule keeps exactly the
distribution it is given; [R] Pitfalls: a top-p that differs between p and q quietly breaks the
identical-distribution guarantee, so both get the same filter. The pages name top-p without a
formula; the reading pinned here is the usual one: top-k keeps the tokens whose logit is at least
the k-th largest, top-p keeps a token when the mass of the strictly larger logits is below top_p,
ties go together, the kept mass is renormalised.
"""
import numpy as np
import pytest
from scipy import special, stats

from _parity import TOL, compare
from oracle.spec_verify_oracle import (filtered_softmax, inverse_cdf, oracle_verify,
                                       temperature_softmax)
from workloads import bf16_round


def softmax_T(z, T):
    return special.softmax(np.asarray(z, np.float64) / np.float64(T))


def rank_definition(z, k):
    """Brute force: token v survives top-k when fewer than k tokens have a strictly larger logit."""
    z = np.asarray(z, np.float64)
    return np.array([np.sum(z > z[v]) < k for v in range(z.size)])


def mass_definition(z, p, top_p):
    """Brute force: token v survives top-p when the mass of the strictly larger logits is below
    top_p (p already renormalised over the top-k set, zero outside it)."""
    z = np.asarray(z, np.float64)
    return np.array([p[v] > 0 and np.sum(p[z > z[v]]) < top_p for v in range(z.size)])


# ------------------------------------------------------------------------------------------------
# Oracle pins (CPU)
# ------------------------------------------------------------------------------------------------

def test_worked_example_by_hand():
    """p = (0.5, 0.3, 0.15, 0.05): cumulative masses 0.5, 0.8, 0.95, 1.0. top_p = 0.79 keeps the
    first two, renormalised to (0.625, 0.375); top_p = 0.81 also keeps the third (/0.95); top_k = 3
    drops the last; top_k = 2 with top_p = 0.7 renormalises to (0.625, 0.375) first, where 0.625 <
    0.7 still admits the second token."""
    p = np.array([0.5, 0.3, 0.15, 0.05])
    z = np.log(p)
    w, m = filtered_softmax(z, 1.0, 0, 0.79)
    assert np.allclose(w, [0.625, 0.375, 0.0, 0.0], atol=1e-15)
    assert m == pytest.approx(0.01, abs=1e-12)
    w, _ = filtered_softmax(z, 1.0, 0, 0.81)
    assert np.allclose(w, [0.5 / 0.95, 0.3 / 0.95, 0.15 / 0.95, 0.0], atol=1e-15)
    w, m = filtered_softmax(z, 1.0, 3, 1.0)
    assert np.allclose(w, [0.5 / 0.95, 0.3 / 0.95, 0.15 / 0.95, 0.0], atol=1e-15)
    assert m == 1.0
    w, _ = filtered_softmax(z, 1.0, 2, 0.7)
    assert np.allclose(w, [0.625, 0.375, 0.0, 0.0], atol=1e-15)
    w, _ = filtered_softmax(z, 1.0, 2, 0.6)
    assert np.allclose(w, [1.0, 0.0, 0.0, 0.0], atol=1e-15)


def test_against_brute_force_definitions():
    rng = np.random.default_rng(1)
    for trial in range(400):
        V = int(rng.integers(1, 30))
        z = rng.standard_normal(V) * 2.0
        if trial % 3 == 0:
            z = np.round(z)                       # ties across the boundaries
        if trial % 7 == 0:
            z[rng.random(V) < 0.3] = -np.inf
            z[0] = 0.5
        T = float(rng.uniform(0.3, 2.0))
        k = int(rng.integers(0, V + 2))
        top_p = float(rng.choice([1.0, rng.uniform(0.01, 1.0)]))
        w, _ = filtered_softmax(z, T, k, top_p)
        p = softmax_T(z, T)
        keep = rank_definition(z, k) if 0 < k < V else np.ones(V, bool)
        pk = np.where(keep, p, 0.0)
        pk /= pk.sum()
        if top_p < 1.0:
            keep &= mass_definition(z, pk, top_p)
        want = np.where(keep, p, 0.0)
        want /= want.sum()
        assert np.allclose(w, want, rtol=1e-12, atol=1e-15), (z, T, k, top_p)
        assert w.sum() == pytest.approx(1.0, abs=1e-12)


def test_degenerate_settings():
    rng = np.random.default_rng(2)
    z = rng.standard_normal(50)
    base = temperature_softmax(z, 0.8)
    for k, tp in ((0, 1.0), (50, 1.0), (51, 1.0), (-3, 1.0), (0, 1.5)):
        w, m = filtered_softmax(z, 0.8, k, tp)
        assert np.array_equal(w, base) and m == 1.0
    # top_k = 1 and a tiny top_p keep the argmax alone
    for k, tp in ((1, 1.0), (0, 1e-9)):
        w, _ = filtered_softmax(z, 0.8, k, tp)
        assert np.array_equal(w, np.eye(50)[np.argmax(z)])
    # all logits equal: every token ties with the k-th and with the top group, so all are kept
    zz = np.full(9, 1.25)
    for k, tp in ((3, 1.0), (0, 0.5), (1, 0.01)):
        w, _ = filtered_softmax(zz, 1.0, k, tp)
        assert np.allclose(w, np.full(9, 1 / 9), atol=1e-15)


def test_margin_is_the_distance_to_the_nearest_boundary():
    z = np.log(np.array([0.4, 0.4, 0.2]))       # groups: {0, 1} (0.8), {2} (0.2)
    _, m = filtered_softmax(z, 1.0, 0, 0.75)
    assert m == pytest.approx(0.05, abs=1e-12)   # |0.8 - 0.75|
    _, m = filtered_softmax(z, 1.0, 0, 0.9)
    assert m == pytest.approx(0.1, abs=1e-12)    # min(|0.8 - 0.9|, |1.0 - 0.9|)


def test_filters_off_give_the_plain_rule():
    rng = np.random.default_rng(3)
    B, G, V = 6, 4, 40
    zt = rng.standard_normal((B, G + 1, V)) * 2
    zd = zt[:, :G] + rng.standard_normal((B, G, V))
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    T[0] = 0.0
    u = rng.random((B, G + 2)).astype(np.float32)
    a = oracle_verify(zt, zd, x, None, T, u)
    o = oracle_verify(zt, zd, x, None, T, u, top_k=np.array([0, V, V + 3, -1, 0, V]),
                      top_p=np.array([1.0, 1.0, 2.0, 1.0, 1.0, 1.0], np.float32))
    for name in ("out_tokens", "out_num_emitted", "out_alpha", "out_p_draft", "out_q_draft"):
        assert np.array_equal(getattr(a, name), getattr(o, name)), name


def test_filtered_quantities():
    """alpha = sum min(p~, q~), p~(x), q~(x) and the bonus drawn from the filtered target."""
    rng = np.random.default_rng(4)
    V = 30
    zt = rng.standard_normal((1, 2, V)) * 2
    zd = zt[:, :1] + rng.standard_normal((1, 1, V))
    x = np.array([[int(np.argmax(zd[0, 0]))]], np.int32)
    T = np.array([0.9], np.float32)
    u = np.array([[0.0, 0.3, 0.77]], np.float32)        # u[0] = 0: the draft is kept
    o = oracle_verify(zt, zd, x, None, T, u, top_k=np.array([7]), top_p=np.array([0.8], np.float32))
    tp = np.float64(np.float32(0.8))
    p, _ = filtered_softmax(zt[0, 0], T[0], 7, tp)
    q, _ = filtered_softmax(zd[0, 0], T[0], 7, tp)
    assert o.out_alpha[0, 0] == pytest.approx(np.minimum(p, q).sum(), abs=1e-14)
    assert o.out_p_draft[0, 0] == pytest.approx(p[x[0, 0]], abs=1e-14)
    assert o.out_q_draft[0, 0] == pytest.approx(q[x[0, 0]], abs=1e-14)
    pb, _ = filtered_softmax(zt[0, 1], T[0], 7, tp)
    assert o.out_num_emitted[0] == 2
    assert o.out_tokens[0, 1] == inverse_cdf(pb, np.float64(u[0, 2]))
    assert pb[o.out_tokens[0, 1]] > 0


@pytest.mark.parametrize("top_p", [0.0, -0.5, np.nan])
def test_row_error_for_an_empty_nucleus(top_p):
    rng = np.random.default_rng(5)
    B, G, V = 3, 2, 12
    zt = rng.standard_normal((B, G + 1, V))
    zd = rng.standard_normal((B, G, V))
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    T = np.array([1.0, 0.0, 1.0], np.float32)            # row 1 greedy: filtering does not apply
    u = rng.random((B, G + 2)).astype(np.float32)
    o = oracle_verify(zt, zd, x, None, T, u, top_p=np.array([top_p, top_p, 1.0], np.float32))
    assert o.out_num_emitted[0] == -1 and (o.out_tokens[0] == -1).all()
    assert o.out_num_emitted[1] >= 1 and o.out_num_emitted[2] >= 1


def test_emitted_token_follows_the_filtered_target():
    """Monte Carlo of the page's guarantee for filtered distributions: drafts drawn from q~, the
    first emitted token follows p~ (chi-square, fixed seed), and nothing outside p~'s support is
    ever emitted."""
    pt = np.array([0.30, 0.25, 0.2, 0.1, 0.08, 0.07])
    pd = np.array([0.1, 0.4, 0.05, 0.3, 0.1, 0.05])
    zt = np.log(pt)[None, None, :].repeat(2, axis=1)
    zd = np.log(pd)[None, None, :]
    k, top_p = 4, np.float32(0.8)
    want, _ = filtered_softmax(zt[0, 0], 1.0, k, np.float64(top_p))
    q, _ = filtered_softmax(zd[0, 0], 1.0, k, np.float64(top_p))
    rng = np.random.default_rng(6)
    N = 20000
    counts = np.zeros(6)
    for _ in range(N):
        x = inverse_cdf(q, rng.random())
        u = rng.random((1, 3)).astype(np.float32)
        o = oracle_verify(zt, zd, np.array([[x]], np.int32), None, np.array([1.0], np.float32), u,
                          top_k=np.array([k]), top_p=np.array([top_p]))
        counts[o.out_tokens[0, 0]] += 1
    assert counts[want == 0].sum() == 0
    s = want > 0
    assert stats.chisquare(counts[s], want[s] * N).pvalue > 1e-3


# ------------------------------------------------------------------------------------------------
# GPU parity through the C ABI
# ------------------------------------------------------------------------------------------------

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_55_gb300 as m
    m.build_library()
    return m


def run_filtered(sv, zt, zd, x, n, T, u, top_k, top_p, dtype):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()   # noqa: E731
    out = sv.verify(dev(zt).to(tdt), dev(zd).to(tdt), dev(x), dev(n), dev(T), dev(u),
                    with_probs=True, top_k=None if top_k is None else dev(top_k),
                    top_p=None if top_p is None else dev(top_p))
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in out]


def check_filtered(zt, zd, x, n, T, u, top_k, top_p, gpu):
    """Parity on every row whose filters are decided farther than the margin from top_p; the rest
    are counted and must still be well formed."""
    o = oracle_verify(zt, zd, x, n, T, u, diagnostics=True, top_k=top_k, top_p=top_p)
    rows = [b for b in range(len(n)) if o.rows[b].filter_margin >= TOL]
    rep = compare(o, *gpu, x, n, rows=rows)
    assert rep.ok(), str(rep)
    for b in set(range(len(n))) - set(rows):
        assert 1 <= gpu[1][b] <= n[b] + 1
    return rep, len(n) - len(rows)


def filter_batch(B, G, V, dtype, seed, greedy_frac=0.15, ties=False):
    """Seeded logits (drafts drawn from the filtered q~ with the oracle's own sampler), ragged
    lengths, per-row top-k from {off, 1, 5, 50, V/2, V-1} and top-p from {off, 0.5, 0.9, 0.99, 1e-3}."""
    rng = np.random.default_rng(seed)
    zt = (rng.standard_normal((B, G + 1, V)) * 2.0).astype(np.float32)
    zd = (zt[:, :G] + rng.standard_normal((B, G, V)).astype(np.float32) * 0.8).astype(np.float32)
    if ties:
        zt, zd = np.round(zt * 2) / 2, np.round(zd * 2) / 2
    if dtype == "bf16":
        zt, zd = bf16_round(zt), bf16_round(zd)
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    T[rng.random(B) < greedy_frac] = 0.0
    n = rng.integers(0, G + 1, B).astype(np.int32)
    n[0] = G
    top_k = rng.choice(np.array([0, 1, 5, 50, V // 2, V - 1], np.int64), B).astype(np.int32)
    top_p = rng.choice(np.array([1.0, 0.5, 0.9, 0.99, 1e-3], np.float32), B).astype(np.float32)
    u = rng.random((B, G + 2), dtype=np.float32)
    x = np.full((B, G), -1, np.int32)
    for b in range(B):
        for i in range(n[b]):
            if T[b] == 0:
                x[b, i] = int(np.argmax(zd[b, i]))
            else:
                q, _ = filtered_softmax(zd[b, i], T[b], int(top_k[b]), np.float64(top_p[b]))
                x[b, i] = inverse_cdf(q, rng.random())
        zt[b, n[b] + 1:] = np.nan
        zd[b, n[b]:] = np.nan
    return zt, zd, x, n, T, u, top_k, top_p


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,V,B,G", [("f32", 256, 16, 4), ("bf16", 1000, 16, 4),
                                         ("f32", 4100, 12, 5), ("bf16", 32000, 12, 4),
                                         ("bf16", 128256, 6, 3), ("f32", 152064, 4, 3)])
def test_gpu_filtered_random_batches(sv, dtype, V, B, G):
    args = filter_batch(B, G, V, dtype, seed=V + B)
    gpu = run_filtered(sv, *args, dtype)
    rep, skipped = check_filtered(*args, gpu)
    print(f"{dtype} V={V}: {rep} filter-margin rows={skipped}")


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gpu_filtered_ties_and_degenerate_rows(sv, dtype):
    """Heavy ties at the top-k boundary and inside the nucleus, rows of equal logits, rows with
    -inf logits (fewer finite logits than k), and top-p / top-k at their extremes."""
    B, G, V = 12, 3, 5000
    zt, zd, x, n, T, u, top_k, top_p = filter_batch(B, G, V, dtype, seed=7, greedy_frac=0.0,
                                                    ties=True)
    zt[1, :2] = 0.75                       # equal logits: every filter keeps every token
    zd[1, :2] = 0.75
    top_k[1], top_p[1] = 3, np.float32(0.5)
    zt[2, 0, 100:] = -np.inf               # only 100 finite logits at position 0, k beyond them
    zd[2, 0, 100:] = -np.inf
    top_k[2], top_p[2] = 300, np.float32(1.0)
    top_k[3], top_p[3] = 1, np.float32(1.0)
    top_k[4], top_p[4] = V - 1, np.float32(0.999999)
    top_k[5], top_p[5] = 0, np.float32(1e-7)
    for b in (1, 2, 3, 4, 5):
        n[b] = G
        zt_b = zt[b, :n[b] + 1]
        zt_b[np.isnan(zt_b)] = 0.0
        zd_b = zd[b, :n[b]]
        zd_b[np.isnan(zd_b)] = 0.0
        for i in range(n[b]):
            q, _ = filtered_softmax(zd[b, i], T[b], int(top_k[b]), np.float64(top_p[b]))
            x[b, i] = inverse_cdf(q, 0.37)
    gpu = run_filtered(sv, zt, zd, x, n, T, u, top_k, top_p, dtype)
    check_filtered(zt, zd, x, n, T, u, top_k, top_p, gpu)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gpu_filtered_token_outside_both_kept_sets(sv, dtype):
    """A drafted token that top-k leaves out of both the filtered p and q has p~(x) = q~(x) = 0: it is
    rejected and never emitted ([R] Why the output is exactly the target's: the filters are applied
    to p and q alike; The output distribution is exactly the target's). Rows 0-3 draft such a
    token; rows 4-7 draft the largest logit (kept by both)."""
    B, G, V = 8, 2, 4096
    rng = np.random.default_rng(77)
    zt = (rng.standard_normal((B, G + 1, V)) * 2.0).astype(np.float32)
    zd = (zt[:, :G] + rng.standard_normal((B, G, V)).astype(np.float32) * 0.3).astype(np.float32)
    if dtype == "bf16":
        zt, zd = bf16_round(zt), bf16_round(zd)
    T = np.ones(B, np.float32)
    n = np.full(B, G, np.int32)
    top_k = np.full(B, 20, np.int32)
    top_p = np.ones(B, np.float32)
    u = rng.random((B, G + 2), dtype=np.float32)
    u[:, :G] = 0.5                          # far from the zero ratio: an exact decision
    x = np.zeros((B, G), np.int32)
    for b in range(B):
        for i in range(G):
            if b < 4:                       # the smallest logit of both rows: outside both top-20 sets
                x[b, i] = int(np.argmin(zt[b, i] + zd[b, i]))
            else:
                x[b, i] = int(np.argmax(zd[b, i]))
    o = oracle_verify(zt, zd, x, n, T, u, diagnostics=True, top_k=top_k, top_p=top_p)
    gpu = run_filtered(sv, zt, zd, x, n, T, u, top_k, top_p, dtype)
    rep = compare(o, *gpu, x, n)
    assert rep.ok(), str(rep)
    for b in range(4):
        assert o.rows[b].k == 0 and gpu[1][b] == 1 and gpu[0][b, 0] != x[b, 0]
        assert gpu[3][b, 0] == 0.0 and gpu[4][b, 0] == 0.0


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,V", [("bf16", 100000), ("f32", 40000)])
def test_gpu_filtered_candidate_lists(sv, dtype, V):
    """Selections the threshold kernel makes by bins and then radix levels over the logits' keys:
    1024 and 1025 ties at the max spread over the row, 1024 ties in the last vectors of the row, a
    k-th largest 57 log2 units below the max (a deep bin), one past 64 log2 units (the tail bin,
    row 0), top-k with top-p, and a bonus-only row."""
    B, G = 8, 3
    rng = np.random.default_rng(V)
    zt = (rng.standard_normal((B, G + 1, V)) * 2.0).astype(np.float32)
    zd = (zt[:, :G] + rng.standard_normal((B, G, V)).astype(np.float32) * 0.8).astype(np.float32)
    T = np.ones(B, np.float32)
    n = np.full(B, G, np.int32)
    top_k = np.array([20, 5, 5, 5, 10, 100, 7, 50], np.int32)
    top_p = np.array([1.0, 1.0, 1.0, 0.9, 1.0, 0.9, 1.0, 0.95], np.float32)
    spread = rng.choice(V, 1025, replace=False)
    zt[1, :, spread[:1024]] = 12.0          # 1024 ties at the max, every chunk
    zd[1, :, spread[:1024]] = 12.0
    zt[2, :, spread] = 12.0                 # 1025 ties
    zd[2, :, spread] = 12.0
    zt[3, :, V - 1024:] = 12.0              # 1024 ties, all in the last chunk
    zd[3, :, V - 1024:] = 12.0
    zt[4] = -40.0                           # three logits at the max, the rest 57 log2 units down
    zd[4] = -40.0
    zt[4, :, [3, V // 2, V - 5]] = 0.0
    zd[4, :, [3, V // 2, V - 5]] = 0.0
    zt[0] = -100.0 + rng.standard_normal((G + 1, V)).astype(np.float32)   # the k-th largest in
    zd[0] = -100.0 + rng.standard_normal((G, V)).astype(np.float32)       # the tail bin
    zt[0, :, [7, V // 3, V - 9]] = 0.0
    zd[0, :, [7, V // 3, V - 9]] = 0.0
    n[6] = 0                                # the bonus position only
    if dtype == "bf16":
        zt, zd = bf16_round(zt), bf16_round(zd)
    u = rng.random((B, G + 2), dtype=np.float32)
    x = np.full((B, G), -1, np.int32)
    for b in range(B):
        for i in range(n[b]):
            q, _ = filtered_softmax(zd[b, i], T[b], int(top_k[b]), np.float64(top_p[b]))
            x[b, i] = inverse_cdf(q, rng.random())
        zt[b, n[b] + 1:] = np.nan
        zd[b, n[b]:] = np.nan
    gpu = run_filtered(sv, zt, zd, x, n, T, u, top_k, top_p, dtype)
    rep, skipped = check_filtered(zt, zd, x, n, T, u, top_k, top_p, gpu)
    assert skipped <= 2, skipped


def smallest_kept(z, T, k, top_p):
    """The smallest logit the oracle's filters keep, for a row of finite logits (every logit has
    probability > 0, so the kept set is where the filtered probability is positive)."""
    assert np.isfinite(z).all()
    pk, _ = filtered_softmax(z, T, int(k), np.float64(top_p))
    return float(np.asarray(z, np.float64)[pk > 0].min())


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,V", [("f32", 4100), ("bf16", 32000), ("bf16", 256000)])
def test_gpu_thresholds_are_the_smallest_kept_logit(sv, dtype, V):
    """spec_verify_filter_thresholds: for every filtered row read by the round, the smallest logit
    the oracle's filters keep (exact: it is one of the row's logits); -inf for greedy rows, rows
    that are not read, rows whose filters are off and rows with a bad top_p."""
    B, G = 10, 3
    zt, zd, x, n, T, u, top_k, top_p = filter_batch(B, G, V, dtype, seed=V + 3, greedy_frac=0.2)
    top_p[B - 1] = 0.0                      # a row error of spec_verify_filtered: -inf
    zt, zd = np.nan_to_num(zt, nan=0.0), np.nan_to_num(zd, nan=0.0)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()   # noqa: E731
    nt = B * (2 * G + 1)
    out = torch.full((nt,), 7.0, dtype=torch.float32, device="cuda")
    sv.spec_verify_filter_thresholds(dev(zt).to(tdt), dev(zd).to(tdt), dev(n), dev(T), dev(top_k),
                                     dev(top_p), out)
    torch.cuda.synchronize()
    tau = out.cpu().numpy()
    checked = 0
    for r in range(nt):
        draft = r >= B * (G + 1)
        b, i = divmod(r - B * (G + 1), G) if draft else divmod(r, G + 1)
        read = i < n[b] if draft else i <= n[b]
        on = (0 < top_k[b] < V) or top_p[b] < 1.0
        if not (read and T[b] > 0 and on and top_p[b] > 0):
            assert tau[r] == -np.inf, (r, tau[r])
            continue
        z = (zd if draft else zt)[b, i]
        _, margin = filtered_softmax(z, T[b], int(top_k[b]), np.float64(top_p[b]))
        if margin < TOL:
            continue
        assert tau[r] == np.float32(smallest_kept(z, T[b], top_k[b], top_p[b])), (r, b, i, tau[r])
        checked += 1
    assert checked >= 5


@pytest.mark.gpu
def test_gpu_filtered_workspace_reused_across_sizes(sv):
    """One workspace serves calls of different sizes: a filtered call leaves every byte of it zero
    (its thresholds lie where another size keeps records and counters), so the next call of other
    sizes on the same workspace still verifies correctly."""
    dtc = sv.SV_DTYPE_F32
    shapes = ((4, 3, 4096, 1), (12, 3, 4096, 2), (3, 8, 4096, 3), (16, 2, 4096, 4))
    # Too small for the kept lists (every row on the streaming kernel), then large enough for them.
    small = sv.spec_verify_workspace_size(64, 8, 4096, dtc)
    assert small < min(sv.spec_verify_filtered_workspace_size(B, G, V, dtc) for B, G, V, _ in shapes)
    large = max(sv.spec_verify_filtered_workspace_size(B, G, V, dtc) for B, G, V, _ in shapes)
    for nbytes, (B, G, V, seed) in [(n, sh) for n in (small, large) for sh in shapes]:
        ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda") if seed == 1 else ws
        zt, zd, x, n, T, u, top_k, top_p = filter_batch(B, G, V, "f32", seed=seed)
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()   # noqa: E731
        outs = (torch.full((B, G + 1), -7, dtype=torch.int32, device="cuda"),
                torch.full((B,), -7, dtype=torch.int32, device="cuda"),
                *[torch.empty((B, G), dtype=torch.float32, device="cuda") for _ in range(3)])
        sv.spec_verify_filtered(dev(zt), dev(zd), dev(x), dev(n), dev(T), dev(top_k), dev(top_p),
                                dev(u), *outs, ws)
        torch.cuda.synchronize()
        assert int(ws.count_nonzero()) == 0, (B, G)
        check_filtered(zt, zd, x, n, T, u, top_k, top_p, [o.cpu().numpy() for o in outs])


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gpu_filtered_bonus_only(sv, dtype):
    """gamma_max = 0: every row is a bonus draw from its filtered target row; top-k rows go through
    the kept lists, the others through the streaming kernel; both against the oracle."""
    B, G, V = 8, 0, 4096
    rng = np.random.default_rng(31)
    zt = (rng.standard_normal((B, 1, V)) * 2.0).astype(np.float32)
    if dtype == "bf16":
        zt = bf16_round(zt)
    zd = np.zeros((B, 0, V), np.float32)
    x = np.zeros((B, 0), np.int32)
    n = np.zeros(B, np.int32)
    T = np.ones(B, np.float32)
    T[7] = 0.0                                    # a greedy row
    top_k = np.array([5, 50, 0, 0, 1, 200, 5, 5], np.int32)
    top_p = np.array([1.0, 0.9, 0.9, 1.0, 1.0, 1.0, 1e-3, 0.5], np.float32)
    u = rng.random((B, 2), dtype=np.float32)
    gpu = run_filtered(sv, zt, zd, x, n, T, u, top_k, top_p, dtype)
    check_filtered(zt, zd, x, n, T, u, top_k, top_p, gpu)
    assert (gpu[1] == 1).all()


@pytest.mark.gpu
def test_gpu_filtered_row_errors(sv):
    B, G, V = 6, 2, 2048
    zt, zd, x, n, T, u, top_k, top_p = filter_batch(B, G, V, "f32", seed=8, greedy_frac=0.0)
    n[:] = G
    for b in range(B):
        for i in range(G):
            x[b, i] = int(np.argmax(zd[b, i]))
    zt[:, :] = np.where(np.isnan(zt), 0.0, zt)
    zd[:, :] = np.where(np.isnan(zd), 0.0, zd)
    top_p[0], top_p[1], top_p[2] = 0.0, -1.0, np.nan
    T[3], top_p[3] = 0.0, 0.0             # greedy row: top-p does not apply
    gpu = run_filtered(sv, zt, zd, x, n, T, u, top_k, top_p, "f32")
    assert (gpu[1][:3] == -1).all() and gpu[1][3] >= 1
    check_filtered(zt, zd, x, n, T, u, top_k, top_p, gpu)


@pytest.mark.gpu
def test_gpu_filters_off_match_the_plain_kernel(sv):
    """Filters off in every row (thresholds -inf) and top_k / top_p None both match the plain
    oracle."""
    B, G, V = 16, 4, 32000
    zt, zd, x, n, T, u, _, _ = filter_batch(B, G, V, "bf16", seed=9)
    a = run_filtered(sv, zt, zd, x, n, T, u, np.zeros(B, np.int32), np.ones(B, np.float32), "bf16")
    b = run_filtered(sv, zt, zd, x, n, T, u, None, None, "bf16")
    o = oracle_verify(zt, zd, x, n, T, u, diagnostics=True)
    for g in (a, b):
        rep = compare(o, *g, x, n)
        assert rep.ok(), str(rep)


@pytest.mark.gpu
def test_gpu_filtered_full_size_sampled_rows(sv):
    """The benchmark's filtered step (B=1024, ragged, V=256000 bf16, seeded top-k / top-p per row)
    in one launch; the oracle checks a sample of rows."""
    from workloads import filter_params, make_workload
    w = make_workload(5, backend="torch", device="cuda")
    top_k, top_p = filter_params(w.B, w.cfg.seed)
    t = w.device_tensors()
    out = sv.verify(t["target_logits"], t["draft_logits"], t["draft_tokens"], t["draft_len"],
                    t["temperature"], t["uniforms"], with_probs=True,
                    top_k=torch.from_numpy(top_k).cuda(), top_p=torch.from_numpy(top_p).cuda())
    torch.cuda.synchronize()
    gpu = [o.cpu().numpy() for o in out]
    rows = sorted({0, w.B - 1, *np.flatnonzero(w.temperature == 0)[:2].tolist(),
                   *np.random.default_rng(10).integers(w.B, size=14).tolist()})
    idx = np.asarray(rows)
    zt = np.stack([w.host_rows(b)[0] for b in rows])
    zd = np.stack([w.host_rows(b)[1] for b in rows])
    check_filtered(zt, zd, w.draft_tokens[idx], w.draft_len[idx], w.temperature[idx],
                   w.uniforms[idx], top_k[idx], top_p[idx], [a[idx] for a in gpu])
    num = gpu[1]
    assert ((num >= 1) & (num <= w.draft_len + 1)).all()
