"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the same seeded inputs.

Every test here needs a GB300 (sm_103a) and is marked gpu.
"""
import numpy as np
import pytest

from _parity import compare, full_batch_parity
from oracle.spec_verify_oracle import oracle_verify, sample_drafts
from workloads import bf16_round, make_workload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_55_gb300 as m
    m.build_library()
    return m


def run_gpu(sv, tensors):
    out = sv.verify(tensors["target_logits"], tensors["draft_logits"], tensors["draft_tokens"],
                    tensors["draft_len"], tensors["temperature"], tensors["uniforms"],
                    with_probs=True)
    torch.cuda.synchronize()
    zt = tensors["target_logits"]
    B, G1, V = zt.shape
    dcode = sv.SV_DTYPE_BF16 if zt.dtype == torch.bfloat16 else sv.SV_DTYPE_F32
    ws = sv.workspace_for(B, G1 - 1, V, dcode, zt.device)
    assert sv.spec_verify_workspace_status(ws, B, G1 - 1) == 0, "a bounded wait gave up"
    return [o.cpu().numpy() for o in out]


def check(oracle_res, gpu, tokens, draft_len, rows=None):
    rep = compare(oracle_res, *gpu, tokens, draft_len, rows=rows)
    assert rep.ok(), str(rep)
    return rep


def host_subset(w, rows):
    """Host arrays of the selected rows (exact stored values) for the oracle."""
    zt = np.stack([w.host_rows(b)[0] for b in rows])
    zd = np.stack([w.host_rows(b)[1] for b in rows])
    idx = np.asarray(rows)
    return zt, zd, w.draft_tokens[idx], w.draft_len[idx], w.temperature[idx], w.uniforms[idx]


# ------------------------------------------------------------------------------------------------
# The five workloads
# ------------------------------------------------------------------------------------------------

def test_config1_full(sv):
    w = make_workload(1, draft_sampler=sample_drafts)
    gpu = run_gpu(sv, w.device_tensors())
    o = oracle_verify(w.target_logits, w.draft_logits, w.draft_tokens, w.draft_len,
                      w.temperature, w.uniforms, diagnostics=True)
    check(o, gpu, w.draft_tokens, w.draft_len)


@pytest.mark.parametrize("cfg", [2, 3])
def test_config_full(sv, cfg):
    w = make_workload(cfg)
    gpu = run_gpu(sv, w.device_tensors())
    o = oracle_verify(w.target_logits, w.draft_logits, w.draft_tokens, w.draft_len,
                      w.temperature, w.uniforms, diagnostics=True)
    rep = check(o, gpu, w.draft_tokens, w.draft_len)
    print(f"config {cfg}: {rep}")


@pytest.mark.parametrize("cfg", [4, 5])
def test_config_full_size_every_row(sv, cfg):
    """The full-size launch (the benchmark's configuration) compared with the oracle on every row,
    under the margin rule; the margin rows and margin positions are counted and printed."""
    w = make_workload(cfg, backend="torch", device="cuda")
    gpu = run_gpu(sv, w.device_tensors())
    rep = full_batch_parity(w, gpu)
    print(f"config {cfg} every row: {rep}")
    assert rep.rows == w.B
    assert rep.ok(), str(rep)
    assert rep.exact_rows + rep.margin_rows + rep.error_rows == w.B


# ------------------------------------------------------------------------------------------------
# Edge shapes and cases
# ------------------------------------------------------------------------------------------------

def small_inputs(B, G, V, dtype, seed, greedy_frac=0.3, ragged=True, scale=2.0, noise=0.8):
    rng = np.random.default_rng(seed)
    zt = (rng.standard_normal((B, G + 1, V)) * scale).astype(np.float32)
    zd = (zt[:, :G] + rng.standard_normal((B, G, V)) * noise).astype(np.float32)
    if dtype == "bf16":
        zt, zd = bf16_round(zt), bf16_round(zd)
    temperature = rng.uniform(0.5, 1.5, B).astype(np.float32)
    temperature[rng.random(B) < greedy_frac] = 0.0
    draft_len = (rng.integers(0, G + 1, B) if ragged else np.full(B, G)).astype(np.int32)
    u = rng.random((B, G + 2), dtype=np.float32)
    tokens = sample_drafts(zd, temperature, rng.random((B, G), dtype=np.float32)) if G else \
        np.zeros((B, 0), np.int32)
    for b in range(B):
        tokens[b, draft_len[b]:] = -1
        zt[b, draft_len[b] + 1:] = np.nan
        zd[b, draft_len[b]:] = np.nan
    return zt, zd, tokens.astype(np.int32), draft_len, temperature, u


def to_dev(zt, zd, tokens, draft_len, temperature, u, dtype):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return dict(target_logits=torch.from_numpy(zt).cuda().to(tdt),
                draft_logits=torch.from_numpy(zd).cuda().to(tdt),
                draft_tokens=torch.from_numpy(tokens).cuda(),
                draft_len=torch.from_numpy(draft_len).cuda(),
                temperature=torch.from_numpy(temperature).cuda(),
                uniforms=torch.from_numpy(u).cuda())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1, 2, 3, 4, 7, 255, 256, 257, 1000, 4100, 8192, 40961, 70000])
def test_edge_vocab_sizes(sv, dtype, V):
    G = 3
    B = 12 if V < 10000 else 6
    args = small_inputs(B, G, V, dtype, seed=V)
    gpu = run_gpu(sv, to_dev(*args, dtype))
    o = oracle_verify(*args, diagnostics=True)
    check(o, gpu, args[2], args[3])


@pytest.mark.parametrize("G", [0, 1, 8, 64])
def test_edge_draft_widths(sv, G):
    B, V = 5, 300
    args = small_inputs(B, G, V, "bf16", seed=100 + G)
    gpu = run_gpu(sv, to_dev(*args, "bf16"))
    o = oracle_verify(*args, diagnostics=True)
    check(o, gpu, args[2], args[3])


@pytest.mark.parametrize("dtype,V", [("bf16", 100277), ("f32", 151937), ("bf16", 262143)])
def test_unaligned_large_vocabularies(sv, dtype, V):
    """Rows whose byte length is not a multiple of 16 above 65536 logits: the element kernel with 16
    or 32 logits per thread, ragged lengths and a greedy mix, against the oracle."""
    B, G = 6, 3
    args = small_inputs(B, G, V, dtype, seed=V % 1000, greedy_frac=0.3)
    gpu = run_gpu(sv, to_dev(*args, dtype))
    rep = check(oracle_verify(*args, diagnostics=True), gpu, args[2], args[3])
    print(f"{dtype} V={V}: {rep}")


def test_vocabulary_beyond_the_row_limits_is_rejected(sv):
    """V above the element kernel's 262144 logits (rows not of 16-byte multiples) returns
    SV_ERR_BAD_SHAPE before anything is enqueued."""
    B, G, V = 1, 1, 262145
    dev = torch.device("cuda")
    zt = torch.zeros((B, G + 1, V), dtype=torch.float32, device=dev)
    zd = torch.zeros((B, G, V), dtype=torch.float32, device=dev)
    with pytest.raises(sv.SpecVerifyError) as ei:
        sv.verify(zt, zd, torch.zeros((B, G), dtype=torch.int32, device=dev), None,
                  torch.ones((B,), dtype=torch.float32, device=dev),
                  torch.full((B, G + 2), 0.5, dtype=torch.float32, device=dev))
    assert ei.value.status == 2


def test_scalar_path_large_vocab_and_misaligned_base(sv):
    # V * 2 bytes not a multiple of 16: the scalar path with the largest chunk it supports.
    V, G, B = 65535, 2, 3
    args = small_inputs(B, G, V, "bf16", seed=7)
    gpu = run_gpu(sv, to_dev(*args, "bf16"))
    check(oracle_verify(*args, diagnostics=True), gpu, args[2], args[3])
    # 16-byte-multiple rows but bases offset by one element: also the scalar path.
    V = 4096
    args = small_inputs(B, G, V, "f32", seed=8)
    t = to_dev(*args, "f32")
    for key in ("target_logits", "draft_logits"):
        big = torch.empty(t[key].numel() + 1, dtype=torch.float32, device="cuda")
        big[1:] = t[key].reshape(-1)
        t[key] = big[1:].view(t[key].shape)
        assert t[key].data_ptr() % 16 != 0
    gpu = run_gpu(sv, t)
    check(oracle_verify(*args, diagnostics=True), gpu, args[2], args[3])


def test_all_greedy_and_argmax_ties(sv):
    B, G, V = 16, 4, 3000
    rng = np.random.default_rng(5)
    zt = bf16_round(rng.integers(-3, 4, (B, G + 1, V)).astype(np.float32))   # many exact ties
    zd = np.full((B, G, V), np.nan, np.float32)                              # never read
    tokens = np.argmax(zt[:, :G], axis=-1).astype(np.int32)
    flip = rng.random((B, G)) < 0.3
    tokens[flip] = rng.integers(0, V, flip.sum())
    temperature = np.zeros(B, np.float32)
    draft_len = rng.integers(0, G + 1, B).astype(np.int32)
    u = np.full((B, G + 2), np.nan, np.float32)                              # never read
    args = (zt, zd, tokens, draft_len, temperature, u)
    gpu = run_gpu(sv, to_dev(*args, "bf16"))
    check(oracle_verify(*args, diagnostics=True), gpu, tokens, draft_len)


@pytest.mark.parametrize("dtype,V,runs", [("bf16", 32768, [(0, 8192)]),
                                           ("f32", 32768, [(0, 4096), (16384, 20480)])])
def test_leading_neg_inf_runs(sv, dtype, V, runs):
    """Runs of -inf logits at the start of the row's chunks: every thread's first batch of logits
    is -inf and its finite logits come later (a running max of -inf must not poison the sum)."""
    B, G = 6, 3
    zt, zd, _, draft_len, temperature, u = small_inputs(B, G, V, dtype, seed=31, greedy_frac=0.2,
                                                        ragged=False)
    for a, b in runs:
        zt[:, :, a:b] = -np.inf
        zd[:, :, a:b] = -np.inf
    rng = np.random.default_rng(32)
    tokens = sample_drafts(zd, temperature, rng.random((B, G), dtype=np.float32))
    args = (zt, zd, tokens, draft_len, temperature, u)
    gpu = run_gpu(sv, to_dev(*args, dtype))
    check(oracle_verify(*args, diagnostics=True), gpu, tokens, draft_len)
    assert (gpu[1] >= 1).all()


def test_zero_draft_mass_and_equal_rows(sv):
    B, G, V = 6, 3, 512
    rng = np.random.default_rng(9)
    zt = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
    zd = zt[:, :G].copy()
    tokens = rng.integers(0, V, (B, G)).astype(np.int32)
    # rows 0-2: equal p and q (every draft accepted); rows 3-5: draft logit -inf at the drafted token
    for b in range(3, 6):
        for i in range(G):
            zd[b, i, tokens[b, i]] = -np.inf
    args = (zt, zd, tokens, np.full(B, G, np.int32), np.ones(B, np.float32),
            rng.random((B, G + 2), dtype=np.float32))
    gpu = run_gpu(sv, to_dev(*args, "f32"))
    o = oracle_verify(*args, diagnostics=True)
    check(o, gpu, tokens, args[3])
    assert (gpu[1] == G + 1).all()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [7, 64, 4096, 65536])
def test_zero_residual_mass_fallback(sv, dtype, V):
    """A rejection whose residual max(0, p - q) has zero mass draws from p with u[G], the reading
    the oracle takes for a step the pages leave open ([R] One round, step 4). The rows of
    zero_residual_row reach it in fp64 and in the kernels' fp32 alike: x's logit (-40 target, -39
    draft) vanishes in both normalisers, so p = q away from x and p(x) = q(x) / e. V = 7 runs on
    the element path, the others on the streaming path."""
    from test_oracle import zero_residual_row
    B, G = 6, 1
    zt = np.zeros((B, G + 1, V), np.float32)
    zd = np.zeros((B, G, V), np.float32)
    tokens = np.zeros((B, G), np.int32)
    for b in range(B):
        x = (3 + 5 * b) % V
        a, d, _ = zero_residual_row(V, x=x, seed=b)
        zt[b], zd[b], tokens[b, 0] = a, d, x
    if dtype == "bf16":
        zt, zd = bf16_round(zt), bf16_round(zd)
    u = np.tile(np.array([0.9, 0.05, 0.81], np.float32), (B, 1))
    u[:, 1] = np.linspace(0.05, 0.95, B, dtype=np.float32)        # a spread of residual uniforms
    args = (zt, zd, tokens, np.ones(B, np.int32), np.ones(B, np.float32), u)
    o = oracle_verify(*args, diagnostics=True)
    for b in range(B):                       # the oracle takes the fallback on every row
        p = o.rows[b]
        assert p.k == 0 and p.ratio[0] == pytest.approx(np.exp(-1.0), rel=1e-9)
    gpu = run_gpu(sv, to_dev(*args, dtype))
    rep = check(o, gpu, tokens, args[3])
    if V <= 4096:              # larger V: single-token masses near 1e-5, most draws in the margin
        assert rep.exact_rows >= B - 1, str(rep)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_mass_drafted_token_is_rejected(sv, dtype):
    """A drafted token that both p and q give zero mass (-inf in both logit rows) is rejected and
    never emitted ([R] The output distribution is exactly the target's); a token with q(x) = 0 and
    p(x) > 0 is kept. Streaming path (V = 4096) and element path (V = 1001)."""
    for V in (4096, 1001):
        B, G = 8, 3
        rng = np.random.default_rng(V)
        zt = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
        zd = (zt[:, :G] + rng.normal(0, 0.5, (B, G, V))).astype(np.float32)
        tokens = rng.integers(0, V, (B, G)).astype(np.int32)
        for b in range(B):
            i = b % G
            zd[b, i, tokens[b, i]] = -np.inf
            if b < B // 2:                     # rows 0-3: p(x) = 0 too
                zt[b, i, tokens[b, i]] = -np.inf
        if dtype == "bf16":
            zt, zd = bf16_round(zt), bf16_round(zd)
        u = rng.random((B, G + 2), dtype=np.float32)
        u[:, :G] = 1e-4                        # other drafts kept; the zero ratio rejects, exactly
        args = (zt, zd, tokens, np.full(B, G, np.int32), np.ones(B, np.float32), u)
        o = oracle_verify(*args, diagnostics=True)
        gpu = run_gpu(sv, to_dev(*args, dtype))
        check(o, gpu, tokens, args[3])
        for b in range(B):
            i = b % G
            if b < B // 2:
                assert gpu[1][b] == i + 1 and gpu[0][b, i] != tokens[b, i], b
                assert gpu[3][b, i] == 0.0 and gpu[4][b, i] == 0.0
            else:                              # q(x) = 0 < p(x): ratio 1, never the rejection
                assert gpu[1][b] - 1 != i, b


@pytest.mark.parametrize("case", ["len_neg", "len_big", "T_nan", "T_neg", "T_inf", "T_subnormal",
                                  "tok_neg", "tok_big", "u_one", "u_nan", "nan_logit",
                                  "pinf_logit", "all_ninf", "draft_nan", "greedy_nan"])
def test_row_errors(sv, case):
    B, G, V = 4, 3, 640
    zt, zd, tokens, n, T, u = small_inputs(B, G, V, "f32", seed=3, greedy_frac=0, ragged=False)
    b = 1
    if case == "len_neg":
        n[b] = -1
    elif case == "len_big":
        n[b] = G + 1
    elif case == "T_nan":
        T[b] = np.nan
    elif case == "T_neg":
        T[b] = -0.5
    elif case == "T_inf":
        T[b] = np.inf
    elif case == "T_subnormal":
        T[b] = np.float32(1e-40)
    elif case == "tok_neg":
        tokens[b, 1] = -3
    elif case == "tok_big":
        tokens[b, 2] = V
    elif case == "u_one":
        u[b, G] = 1.0
    elif case == "u_nan":
        u[b, 0] = np.nan
    elif case == "nan_logit":
        zt[b, G, 17] = np.nan
    elif case == "pinf_logit":
        zt[b, 1, 600] = np.inf
    elif case == "all_ninf":
        zt[b, 0, :] = -np.inf
    elif case == "draft_nan":
        zd[b, 2, 300] = np.nan
    elif case == "greedy_nan":
        T[b] = 0.0
        zt[b, 2, 5] = np.nan
    args = (zt, zd, tokens, n, T, u)
    gpu = run_gpu(sv, to_dev(*args, "f32"))
    o = oracle_verify(*args, diagnostics=True)
    assert not o.rows[b].valid
    check(o, gpu, tokens, np.clip(n, 0, G))


def test_determinism_and_workspace_left_zeroed(sv):
    w = make_workload(2)
    t = w.device_tensors()
    a = run_gpu(sv, t)
    b = run_gpu(sv, t)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    from speculative_decoding_verification_55_gb300 import workspace_for, SV_DTYPE_BF16
    ws = workspace_for(w.B, w.G, w.V, SV_DTYPE_BF16, t["target_logits"].device)
    assert int(ws.count_nonzero()) == 0
    from speculative_decoding_verification_55_gb300 import spec_verify_workspace_status
    assert spec_verify_workspace_status(ws, w.B, w.G) == 0


# ------------------------------------------------------------------------------------------------
# Distribution checks on the GPU path
# ------------------------------------------------------------------------------------------------

def test_gpu_emitted_token_distributed_as_target(sv):
    """cgnarendiran.github.io four-token example, one drafted position per row, drafts ~ q: the
    first emitted token follows p (chi-square at a fixed seed)."""
    from scipy import stats
    p = np.array([0.30, 0.40, 0.20, 0.10])
    q = np.array([0.60, 0.20, 0.15, 0.05])
    N = 60000
    rng = np.random.default_rng(2024)
    x = rng.choice(4, size=(N, 1), p=q).astype(np.int32)
    zt = np.broadcast_to(np.log(p).astype(np.float32), (N, 2, 4)).copy()
    zd = np.broadcast_to(np.log(q).astype(np.float32), (N, 1, 4)).copy()
    u = rng.random((N, 3), dtype=np.float32)
    args = (zt, zd, x, np.ones(N, np.int32), np.ones(N, np.float32), u)
    gpu = run_gpu(sv, to_dev(*args, "f32"))
    counts = np.bincount(gpu[0][:, 0], minlength=4)
    assert stats.chisquare(counts, N * p).pvalue > 1e-3, counts
    assert abs(np.mean(gpu[1] == 2) - 0.7) < 4 * np.sqrt(0.21 / N)
    np.testing.assert_allclose(gpu[2][:, 0], 0.7, atol=1e-5)
