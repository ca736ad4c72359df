"""Greedy tree verification (Medusa-style candidate trees): oracle pins on the CPU and GPU parity of
spec_verify_tree_greedy.

[B] "Inference: distillation and speculative decoding" (brunomaga.github.io), Medusa: the top
candidates of the heads form a tree of continuations, verified in one target pass with tree
attention; the root is the target's own next token; a node is accepted when its parent is accepted
and its token is the target's prediction after its parent; the longest accepted path is kept and the
target's prediction after its last node is the next token.
"""
import numpy as np
import pytest

from oracle.spec_verify_oracle import oracle_tree_greedy, oracle_verify
from workloads import bf16_round


def medusa_parents(top_k, heads):
    """Parent list of the tree the page builds: the root, then top_k children for every node of the
    previous level, level by level (parents before children)."""
    parents, level = [-1], [0]
    for _ in range(heads):
        new = []
        for par in level:
            for _ in range(top_k):
                new.append(len(parents))
                parents.append(par)
        level = new
    return np.array(parents, np.int32)


def random_tree(rng, N, V, zt, p_match=0.6):
    par = np.full(N, -1, np.int32)
    for j in range(1, N):
        par[j] = rng.integers(0, j)
    tok = rng.integers(0, V, N).astype(np.int32)
    g = np.argmax(zt, axis=-1)
    for j in range(1, N):
        if rng.random() < p_match:
            tok[j] = g[par[j]]
    return tok, par


def brute_force_path(zt, tok, par, n):
    """Every node's path from the root, kept if each of its nodes matches the argmax at its parent;
    the longest kept path (lowest end node among the longest)."""
    g = [int(np.argmax(zt[j])) for j in range(n)]
    best = [0]
    for j in range(n):
        nodes = [j]
        while nodes[-1] != 0:
            nodes.append(int(par[nodes[-1]]))
        nodes.reverse()
        if all(int(tok[nodes[d]]) == g[nodes[d - 1]] for d in range(1, len(nodes))):
            if len(nodes) > len(best):
                best = nodes
    return best, g[best[-1]]


# ------------------------------------------------------------------------------------------------
# Oracle pins (CPU)
# ------------------------------------------------------------------------------------------------

def test_medusa_example_by_hand():
    """top_k = 2, two heads: nodes 0 | 1 2 | 3 4 (under 1) 5 6 (under 2). The target predicts node
    2's token after the root and node 6's token after node 2: the path is 0 -> 2 -> 6."""
    par = medusa_parents(2, 2)
    assert par.tolist() == [-1, 0, 0, 1, 1, 2, 2]
    V = 8
    zt = np.zeros((7, V))
    pred = [5, 0, 7, 1, 1, 2, 3]             # the target's argmax at each node
    for j, t in enumerate(pred):
        zt[j, t] = 4.0
    tok = np.array([1, 4, 5, 1, 0, 6, 7], np.int32)   # node 2 = 5 = pred[0]; node 6 = 7 = pred[2]
    r = oracle_tree_greedy(zt[None], tok[None], par[None])
    assert r.path[0].tolist() == [0, 2, 6, -1, -1, -1, -1]
    assert r.path_len[0] == 3
    assert r.tokens[0].tolist() == [1, 5, 7, 3, -1, -1, -1, -1]   # path tokens, then pred[6] = 3
    assert r.pred[0].tolist() == pred


def test_against_brute_force_paths():
    rng = np.random.default_rng(11)
    for trial in range(300):
        N = int(rng.integers(1, 20))
        V = int(rng.integers(2, 6))
        zt = rng.standard_normal((N, V))
        if trial % 3 == 0:
            zt = np.round(zt)                   # ties in the argmax
        tok, par = random_tree(rng, N, V, zt)
        n = int(rng.integers(1, N + 1))
        r = oracle_tree_greedy(zt[None], tok[None], par[None], np.array([n]))
        path, nxt = brute_force_path(zt, tok, par, n)
        L = len(path)
        assert r.path_len[0] == L and r.path[0, :L].tolist() == path
        assert r.tokens[0, :L + 1].tolist() == [int(tok[j]) for j in path] + [nxt]


def test_chain_tree_is_the_linear_greedy_rule():
    """A chain (parent j-1) with the root followed by the drafts gives the linear greedy
    verification of the general oracle: path length k + 1 and the same emitted tokens."""
    rng = np.random.default_rng(12)
    for _ in range(100):
        G, V = int(rng.integers(0, 7)), int(rng.integers(2, 7))
        zt = rng.standard_normal((G + 1, V))
        x = rng.integers(0, V, G).astype(np.int32)
        g = np.argmax(zt, axis=-1)
        for i in range(G):
            if rng.random() < 0.7:
                x[i] = g[i]
        root = int(rng.integers(V))
        tok = np.concatenate([[root], x]).astype(np.int32)
        par = np.arange(-1, G, dtype=np.int32)
        r = oracle_tree_greedy(zt[None], tok[None], par[None])
        o = oracle_verify(zt[None], np.zeros((1, G, V)), x[None], None, np.zeros(1, np.float32),
                          np.zeros((1, G + 2), np.float32))
        k = int(o.out_num_emitted[0]) - 1
        assert r.path_len[0] == k + 1
        assert r.tokens[0, :k + 2].tolist() == [root] + o.out_tokens[0, :k + 1].tolist()


def test_deepest_tie_takes_the_lowest_node():
    V = 4
    zt = np.zeros((4, V))
    zt[0, 2] = 1.0                           # the target predicts token 2 after the root
    zt[1, 0] = 1.0
    zt[2, 3] = 1.0
    tok = np.array([0, 2, 2, 1], np.int32)   # nodes 1 and 2 both accepted at depth 1
    par = np.array([-1, 0, 0, 0], np.int32)
    r = oracle_tree_greedy(zt[None], tok[None], par[None])
    assert r.path[0, :2].tolist() == [0, 1] and r.tokens[0, :3].tolist() == [0, 2, 0]


@pytest.mark.parametrize("case", ["size0", "size_big", "root_parent", "parent_ahead", "tok_neg",
                                  "tok_big", "nan", "inf", "all_neg_inf"])
def test_row_errors(case):
    rng = np.random.default_rng(13)
    N, V = 5, 6
    zt = rng.standard_normal((2, N, V))
    tok = rng.integers(0, V, (2, N)).astype(np.int32)
    par = np.tile(np.array([-1, 0, 1, 1, 2], np.int32), (2, 1))
    size = np.array([N, N])
    if case == "size0":
        size[0] = 0
    elif case == "size_big":
        size[0] = N + 1
    elif case == "root_parent":
        par[0, 0] = 0
    elif case == "parent_ahead":
        par[0, 3] = 3
    elif case == "tok_neg":
        tok[0, 2] = -1
    elif case == "tok_big":
        tok[0, 4] = V
    elif case == "nan":
        zt[0, 3, 1] = np.nan
    elif case == "inf":
        zt[0, 1, 0] = np.inf
    else:
        zt[0, 2] = -np.inf
    r = oracle_tree_greedy(zt, tok, par, size)
    assert r.path_len[0] == -1 and (r.path[0] == -1).all() and (r.tokens[0] == -1).all()
    assert r.path_len[1] >= 1


# ------------------------------------------------------------------------------------------------
# GPU parity through the C ABI (integer outputs: bit-exact)
# ------------------------------------------------------------------------------------------------

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_55_gb300 as m
    m.build_library()
    return m


def run_tree(sv, zt, tok, par, size, dtype):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = sv.verify_tree(torch.from_numpy(np.ascontiguousarray(zt)).cuda().to(tdt),
                         torch.from_numpy(tok).cuda(), torch.from_numpy(par).cuda(),
                         None if size is None else torch.from_numpy(size).cuda())
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in out]


def check_tree(r, gpu):
    path, plen, toks, pred = gpu
    assert np.array_equal(plen, r.path_len), (plen, r.path_len)
    assert np.array_equal(path, r.path)
    assert np.array_equal(toks, r.tokens)
    assert np.array_equal(pred, r.pred)


def tree_batch(B, N, V, dtype, seed, medusa=False, full=False):
    rng = np.random.default_rng(seed)
    zt = (rng.standard_normal((B, N, V)) * 2.0).astype(np.float32)
    if dtype == "bf16":
        zt = bf16_round(zt)
    tok = np.zeros((B, N), np.int32)
    par = np.zeros((B, N), np.int32)
    size = rng.integers(1, N + 1, B).astype(np.int32)
    size[0] = N
    if full:
        size[:] = N
    for b in range(B):
        t, p = random_tree(rng, N, V, zt[b])
        if medusa:
            p = medusa_parents(2, int(np.log2(N + 1)) - 1)
            g = np.argmax(zt[b], axis=-1)
            t = np.where(rng.random(N) < 0.7, g[np.maximum(p, 0)], rng.integers(0, V, N))
        tok[b], par[b] = t, p
        zt[b, size[b]:] = np.nan             # nodes beyond the row's size are never read
    return zt, tok, par, size


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,V,N,B", [("f32", 256, 7, 16), ("bf16", 1000, 31, 8),
                                         ("f32", 4100, 65, 4), ("bf16", 32000, 15, 12),
                                         ("bf16", 128256, 31, 6), ("f32", 152064, 5, 3)])
def test_gpu_tree_random(sv, dtype, V, N, B):
    zt, tok, par, size = tree_batch(B, N, V, dtype, seed=V + N)
    gpu = run_tree(sv, zt, tok, par, size, dtype)
    check_tree(oracle_tree_greedy(zt, tok, par, size), gpu)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gpu_tree_medusa_shapes_and_ties(sv, dtype):
    zt, tok, par, size = tree_batch(10, 31, 4096, dtype, seed=5, medusa=True, full=True)
    zt = np.round(zt)                          # many argmax ties
    gpu = run_tree(sv, zt, tok, par, size, dtype)
    check_tree(oracle_tree_greedy(zt, tok, par, size), gpu)
    gpu = run_tree(sv, zt, tok, par, None, dtype)   # tree_size NULL: every row full
    check_tree(oracle_tree_greedy(zt, tok, par, None), gpu)


@pytest.mark.gpu
def test_gpu_tree_row_errors(sv):
    B, N, V = 8, 6, 512
    rng = np.random.default_rng(21)
    zt = rng.standard_normal((B, N, V)).astype(np.float32)
    tok = rng.integers(0, V, (B, N)).astype(np.int32)
    par = np.tile(np.array([-1, 0, 0, 1, 2, 2], np.int32), (B, 1))
    size = np.full(B, N, np.int32)
    size[0] = 0
    size[1] = N + 1
    par[2, 0] = 1
    par[3, 4] = 5
    tok[4, 3] = V
    zt[5, 2, 7] = np.nan
    zt[6, 1] = -np.inf
    gpu = run_tree(sv, zt, tok, par, size, "f32")
    r = oracle_tree_greedy(zt, tok, par, size)
    assert (r.path_len[:7] == -1).all() and r.path_len[7] >= 1
    check_tree(r, gpu)


@pytest.mark.gpu
def test_gpu_tree_workspace_left_zeroed(sv):
    zt, tok, par, size = tree_batch(6, 9, 2048, "f32", seed=3)
    a = run_tree(sv, zt, tok, par, size, "f32")
    b = run_tree(sv, zt, tok, par, size, "f32")
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    ws = sv.workspace_for(6, 8, 2048, sv.SV_DTYPE_F32, torch.device("cuda"))
    assert int(ws.count_nonzero()) == 0
    assert sv.spec_verify_workspace_status(ws, 6, 8) == 0


@pytest.mark.gpu
def test_gpu_tree_full_size_batch(sv):
    """The benchmark's tree batch (B=256 Medusa trees of 31 nodes, V=128256 bf16): enough position
    slots that the streaming path takes its large-chunk clusters. A seeded sample of rows against
    the oracle."""
    import importlib.util
    from pathlib import Path
    spec = importlib.util.spec_from_file_location(
        "bench_for_tree", Path(__file__).resolve().parent.parent / "bench.py")
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    zt, tok, par = bench.tree_inputs(bench.TREE_B, 7, "torch")
    out = sv.verify_tree(zt, tok, par, None)
    torch.cuda.synchronize()
    gpu = [o.cpu().numpy() for o in out]
    rows = np.sort(np.random.default_rng(11).choice(bench.TREE_B, 16, replace=False))
    idx = torch.from_numpy(rows).cuda()
    r = oracle_tree_greedy(zt[idx].float().cpu().numpy(), tok[idx].cpu().numpy(),
                           par[idx].cpu().numpy())
    check_tree(r, [g[rows] for g in gpu])
