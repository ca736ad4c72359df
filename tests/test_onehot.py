"""One-hot drafts (a greedy drafter): oracle pins on the CPU and GPU parity of spec_verify_onehot.

[B] "Inference: distillation and speculative decoding" (brunomaga.github.io), Draft-model speculative
decoding: greedy drafts are the special case of a one-hot draft distribution; the target keeps the
draft x with probability p(x) and on a rejection samples from p without x, which still yields
tokens distributed as p. [R] "Speculative decoding" (rayaq.ca), One round, steps 3-5.
"""
import numpy as np
import pytest
from scipy import special, stats

from _parity import compare
from oracle.spec_verify_oracle import oracle_verify, oracle_verify_onehot, onehot_draft_logits
from workloads import bf16_round, make_workload


def softmax_T(z, T):
    return special.softmax(np.asarray(z, np.float64) / np.float64(T))


# ------------------------------------------------------------------------------------------------
# Oracle pins (CPU)
# ------------------------------------------------------------------------------------------------

def test_onehot_draft_logits_give_a_point_mass():
    zd = onehot_draft_logits(np.array([2, 0, 7]), 3, 5)
    assert np.array_equal(softmax_T(zd[0], 0.7), np.eye(5)[2])
    assert np.array_equal(softmax_T(zd[1], 1.3), np.eye(5)[0])
    assert np.all(zd[2] == -np.inf)           # out-of-range token: nothing to put the mass on


def test_alpha_is_p_of_x_and_q_is_one():
    """Closed forms: sum_v min(p(v), [v == x]) = p(x); q(x) = 1."""
    rng = np.random.default_rng(1)
    B, G, V = 6, 4, 37
    zt = rng.standard_normal((B, G + 1, V)) * 2
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    u = rng.random((B, G + 2)).astype(np.float32)
    o = oracle_verify_onehot(zt, x, np.full(B, G), T, u)
    for b in range(B):
        for i in range(G):
            p = softmax_T(zt[b, i], T[b])
            assert o.out_alpha[b, i] == pytest.approx(p[x[b, i]], abs=1e-15)
            assert o.out_p_draft[b, i] == pytest.approx(p[x[b, i]], abs=1e-15)
            assert o.out_q_draft[b, i] == 1.0


def test_accept_iff_u_below_p_of_x():
    """One drafted position: kept exactly when u < p(x) (min(1, p/q) with q(x) = 1)."""
    rng = np.random.default_rng(2)
    V = 11
    zt = rng.standard_normal((1, 2, V))
    x = np.array([[4]], np.int32)
    px = softmax_T(zt[0, 0], 1.0)[4]
    for du, kept in ((-1e-4, True), (+1e-4, False)):
        u = np.array([[px + du, 0.3, 0.6]], np.float32)
        o = oracle_verify_onehot(zt, x, np.array([1]), np.array([1.0], np.float32), u)
        assert (o.out_num_emitted[0] == 2) == kept


def test_residual_draw_is_p_without_x():
    """On a rejection the replacement is the inverse CDF (strict >) of p with x's mass removed."""
    rng = np.random.default_rng(3)
    V = 23
    for trial in range(50):
        zt = rng.standard_normal((1, 2, V)) * 1.5
        x = int(rng.integers(V))
        p = softmax_T(zt[0, 0], 1.0)
        u_res = np.float32(rng.random())
        u = np.array([[1.0 - 1e-7, u_res, 0.5]], np.float32)     # u[0] >= p(x): rejected
        o = oracle_verify_onehot(zt, np.array([[x]], np.int32), np.array([1]),
                                 np.array([1.0], np.float32), u)
        w = p.copy()
        w[x] = 0.0
        c = np.cumsum(w)
        want = int(np.argmax(c > np.float64(u_res) * c[-1]))
        assert o.out_num_emitted[0] == 1 and o.out_tokens[0, 0] == want != x


def test_greedy_rows_unchanged():
    """Temperature 0 rows are verified by argmax match whatever the draft distribution."""
    rng = np.random.default_rng(4)
    B, G, V = 5, 3, 17
    zt = rng.standard_normal((B, G + 1, V))
    zd = rng.standard_normal((B, G, V))
    x = np.argmax(zt[:, :G], axis=-1).astype(np.int32)
    x[1, 1] = (x[1, 1] + 1) % V
    T = np.zeros(B, np.float32)
    u = rng.random((B, G + 2)).astype(np.float32)
    a = oracle_verify(zt, zd, x, None, T, u)
    o = oracle_verify_onehot(zt, x, None, T, u)
    assert np.array_equal(a.out_tokens, o.out_tokens) and np.array_equal(a.out_num_emitted,
                                                                         o.out_num_emitted)


def test_first_token_distributed_as_target():
    """Monte Carlo ([B]: still yields tokens distributed as p): with a fixed greedy draft x and
    random u, the first emitted token follows p (chi-square, fixed seed)."""
    p = np.array([0.05, 0.4, 0.25, 0.2, 0.1])
    zt = np.log(p)[None, None, :].repeat(2, axis=1)
    x = np.array([[1]], np.int32)
    rng = np.random.default_rng(5)
    N = 20000
    counts = np.zeros(5)
    for _ in range(N):
        u = rng.random((1, 3)).astype(np.float32)
        o = oracle_verify_onehot(zt, x, np.array([1]), np.array([1.0], np.float32), u)
        counts[o.out_tokens[0, 0]] += 1
    assert stats.chisquare(counts, p * N).pvalue > 1e-3


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


def run_onehot(sv, t):
    out = sv.verify(t["target_logits"], None, t["draft_tokens"], t["draft_len"], t["temperature"],
                    t["uniforms"], with_probs=True, onehot=True)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in out]


def dev_inputs(zt, tokens, draft_len, T, u, dtype):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return dict(target_logits=torch.from_numpy(np.ascontiguousarray(zt)).cuda().to(tdt),
                draft_tokens=torch.from_numpy(tokens).cuda(),
                draft_len=torch.from_numpy(draft_len).cuda(),
                temperature=torch.from_numpy(T).cuda(),
                uniforms=torch.from_numpy(u).cuda())


def check(o, gpu, tokens, draft_len, rows=None):
    rep = compare(o, *gpu, tokens, draft_len, rows=rows)
    assert rep.ok(), str(rep)
    return rep


def random_batch(B, G, V, dtype, seed, greedy_frac=0.2):
    rng = np.random.default_rng(seed)
    zt = (rng.standard_normal((B, G + 1, V)) * 2.0).astype(np.float32)
    if dtype == "bf16":
        zt = bf16_round(zt)
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    T[rng.random(B) < greedy_frac] = 0.0
    draft_len = rng.integers(0, G + 1, B).astype(np.int32)
    # greedy drafts of a noisy copy of the target (a typical one-hot drafter), some random tokens
    x = np.argmax(zt[:, :G] + rng.standard_normal((B, G, V)).astype(np.float32), axis=-1)
    x = np.where(rng.random((B, G)) < 0.3, rng.integers(0, V, (B, G)), x).astype(np.int32)
    u = rng.random((B, G + 2), dtype=np.float32)
    for b in range(B):
        x[b, draft_len[b]:] = -1
        zt[b, draft_len[b] + 1:] = np.nan
    return zt, x, draft_len, T, u


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,V", [("f32", 256), ("bf16", 1000), ("f32", 4100), ("bf16", 8192),
                                     ("bf16", 70000), ("f32", 152064)])
def test_gpu_onehot_random_batches(sv, dtype, V):
    B, G = (12, 5) if V < 100000 else (4, 3)
    zt, x, n, T, u = random_batch(B, G, V, dtype, seed=V)
    gpu = run_onehot(sv, dev_inputs(zt, x, n, T, u, dtype))
    o = oracle_verify_onehot(zt, x, n, T, u, diagnostics=True)
    check(o, gpu, x, n)


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", [2, 3])
def test_gpu_onehot_configs(sv, cfg):
    w = make_workload(cfg)
    t = w.device_tensors()
    gpu = run_onehot(sv, t)
    o = oracle_verify_onehot(w.target_logits, w.draft_tokens, w.draft_len, w.temperature,
                             w.uniforms, diagnostics=True)
    rep = check(o, gpu, w.draft_tokens, w.draft_len)
    print(f"one-hot config {cfg}: {rep}")


@pytest.mark.gpu
def test_gpu_onehot_full_size_sampled_rows(sv):
    """The benchmark shape (B=1024, ragged, V=256000 bf16) in one launch; the oracle checks rows."""
    w = make_workload(5, backend="torch", device="cuda")
    gpu = run_onehot(sv, w.device_tensors())
    rows = sorted({0, w.B - 1, *np.flatnonzero(w.temperature == 0)[:2].tolist(),
                   *np.random.default_rng(9).integers(w.B, size=20).tolist()})
    zt = np.stack([w.host_rows(b)[0] for b in rows])
    idx = np.asarray(rows)
    o = oracle_verify_onehot(zt, w.draft_tokens[idx], w.draft_len[idx], w.temperature[idx],
                             w.uniforms[idx], diagnostics=True)
    check(o, [a[rows] for a in gpu], w.draft_tokens[rows], w.draft_len[rows])
    num = gpu[1]
    assert ((num >= 1) & (num <= w.draft_len + 1)).all()


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gpu_onehot_edge_tokens(sv, dtype):
    """x at the row maximum, x with a -inf logit (never kept), x carrying almost all the mass, x at
    chunk edges (the first and last vector of a chunk), and a drafted token out of range."""
    B, G, V = 8, 2, 70000
    rng = np.random.default_rng(77)
    zt = (rng.standard_normal((B, G + 1, V)) * 2.0).astype(np.float32)
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    x[0, 0] = int(np.argmax(zt[0, 0]))
    zt[1, 0, x[1, 0]] = -np.inf
    zt[2, 0, x[2, 0]] = 40.0
    E = 8 if dtype == "bf16" else 4
    x[3, 0], x[3, 1] = 0, V - 1
    x[4, 0] = 2048 * E - 1                 # last element of a 16 KB slot / chunk region
    x[4, 1] = 2048 * E
    x[5, 0] = V                            # out of range: row error
    if dtype == "bf16":
        zt = bf16_round(zt)
        zt[1, 0, x[1, 0]] = -np.inf
    n = np.full(B, G, np.int32)
    T = np.ones(B, np.float32)
    u = rng.random((B, G + 2), dtype=np.float32)
    u[:, 0] = 0.999                        # mostly rejected: exercise the residual draws
    gpu = run_onehot(sv, dev_inputs(zt, x, n, T, u, dtype))
    o = oracle_verify_onehot(zt, x, n, T, u, diagnostics=True)
    check(o, gpu, x, n)
    assert gpu[1][5] == -1
    assert gpu[0][1, 0] != x[1, 0]          # a -inf draft is never kept nor redrawn


@pytest.mark.gpu
def test_gpu_onehot_rejects_unsupported_rows(sv):
    t = dev_inputs(np.zeros((2, 2, 10), np.float32), np.zeros((2, 1), np.int32),
                   np.ones(2, np.int32), np.ones(2, np.float32), np.zeros((2, 3), np.float32), "f32")
    with pytest.raises(sv.SpecVerifyError) as ei:
        run_onehot(sv, t)
    assert "BAD_SHAPE" in str(ei.value)


@pytest.mark.gpu
def test_gpu_onehot_first_token_distributed_as_target(sv):
    """Monte Carlo on the GPU: N rows with the same p and the same greedy draft x; the emitted first
    token follows p (chi-square at a fixed seed)."""
    p = np.array([0.05, 0.4, 0.25, 0.2, 0.1, 0.0, 0.0, 0.0])
    with np.errstate(divide="ignore"):
        lp = np.log(p).astype(np.float32)
    N = 50000
    zt = np.broadcast_to(lp, (N, 2, 8)).copy()
    x = np.full((N, 1), 1, np.int32)
    rng = np.random.default_rng(6)
    u = rng.random((N, 3), dtype=np.float32)
    gpu = run_onehot(sv, dev_inputs(zt, x, np.ones(N, np.int32), np.ones(N, np.float32), u, "f32"))
    counts = np.bincount(gpu[0][:, 0], minlength=8)[:5]
    assert stats.chisquare(counts, p[:5] * N).pvalue > 1e-3
