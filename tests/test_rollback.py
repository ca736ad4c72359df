"""KV-cache rollback after a round: oracle pins on the CPU and GPU parity of spec_verify_kv_rollback.

[R] "Speculative decoding" (rayaq.ca ml-models), Verification attention and the cache: with k drafts
accepted the target keeps the first n + k + 1 cache entries; the drafter's cache is rolled back the
same way. [B] "Inference: distillation and speculative decoding" (brunomaga.github.io), Draft-model
speculative decoding: the drafter reuses the longest prefix of the tokens it has already processed.
"""
import json
from pathlib import Path

import numpy as np
import pytest

from oracle.spec_verify_oracle import kv_rollback, oracle_verify, sample_drafts

GOLDEN = Path(__file__).resolve().parent / "golden" / "rayaq_cache_rollback.json"


# ------------------------------------------------------------------------------------------------
# Oracle pins (CPU)
# ------------------------------------------------------------------------------------------------

def test_page_example():
    g = json.loads(GOLDEN.read_text())
    n, G, k = g["prefix_entries_before_verification"], g["gamma"], g["drafts_accepted"]
    assert n + G + 1 == g["entries_after_verification"]
    target, _, dropped = kv_rollback([n], [G], [k + 1], None, G)
    assert target[0] == g["entries_kept"]
    assert dropped[0][1] - dropped[0][0] == g["entries_dropped"]


def drafter_prefix(processed, new_tokens):
    """The drafter's reuse rule, restated on token lists: the longest common prefix of the tokens
    its cache holds and the new sequence, excluding the new sequence's last token (always
    processed again)."""
    n = min(len(processed), len(new_tokens) - 1)
    c = 0
    while c < n and processed[c] == new_tokens[c]:
        c += 1
    return c


def test_drafter_keeps_its_valid_prefix():
    """Random sampled and greedy rounds through the oracle: the cache the drafter can reuse, found by
    comparing token lists (it processed the sequence and all drafts but the last), equals
    min(drafter entries, n + k + 1), one entry short on a full accept."""
    rng = np.random.default_rng(31)
    for trial in range(200):
        G, V = int(rng.integers(1, 7)), int(rng.integers(2, 9))
        T = np.float32(0.0 if trial % 4 == 0 else rng.uniform(0.5, 1.5))
        zt = rng.standard_normal((1, G + 1, V)) * 2
        zd = rng.standard_normal((1, G, V)) * 2
        x = sample_drafts(zd, np.array([T]), rng.random((1, G), dtype=np.float32))
        u = rng.random((1, G + 2), dtype=np.float32)
        o = oracle_verify(zt, zd, x, None, np.array([T]), u)
        e = int(o.out_num_emitted[0])
        prefix = list(rng.integers(0, V, int(rng.integers(1, 6))))      # accepted tokens so far
        n = len(prefix) - 1                                            # the target's cache
        processed = prefix + list(x[0, :G - 1])                        # the drafter's cache
        new = prefix + list(o.out_tokens[0, :e])
        target, drafter, dropped = kv_rollback([n], [G], [e], [len(processed)], G)
        assert target[0] == len(new) - 1 == n + e
        assert drafter[0] == drafter_prefix(processed, new)
        assert dropped[0] == (n + e, n + G + 1)


def test_row_error_commits_nothing():
    target, drafter, dropped = kv_rollback([10, 10], [3, 3], [-1, 2], [13, 13], 3)
    assert target.tolist() == [10, 12] and drafter.tolist() == [10, 12]
    assert dropped == [(10, 14), (12, 14)]


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


def run_rollback(sv, n, g, e, d, G, cache=None):
    dev = torch.device("cuda")
    B = len(n)
    t = lambda a: torch.as_tensor(np.asarray(a, np.int32), device=dev)
    tl = torch.full((B,), -7, dtype=torch.int32, device=dev)
    dl = torch.full((B,), -7, dtype=torch.int32, device=dev)
    sv.spec_verify_kv_rollback(t(n), None if g is None else t(g), t(e), None if d is None else t(d),
                               tl, dl, cache=cache, gamma_max=G)
    torch.cuda.synchronize()
    return tl.cpu().numpy(), dl.cpu().numpy()


@pytest.mark.gpu
def test_gpu_lengths_and_dropped_entries_zeroed(sv):
    rng = np.random.default_rng(41)
    B, G, L = 96, 8, 24
    n = rng.integers(0, 14, B)
    g = rng.integers(0, G + 1, B)
    e = np.array([int(rng.integers(1, gi + 2)) for gi in g])
    e[::7] = -1                                   # row errors
    d = n + g + rng.integers(-2, 1, B)
    n[3] = 30                                     # beyond the cache: lengths only, no bytes touched
    cache = torch.randint(1, 255, (B, L, 3, 32), dtype=torch.uint8, device="cuda")   # 96-byte entries
    before = cache.cpu().numpy().copy()
    tl, dl = run_rollback(sv, n, g, e, d, G, cache)
    want_t, want_d, dropped = kv_rollback(n, g, e, d, G)
    assert np.array_equal(tl, want_t) and np.array_equal(dl, want_d)
    after = cache.cpu().numpy()
    for b in range(B):
        lo, hi = dropped[b]
        lo, hi = max(lo, 0), min(hi, L)
        mask = np.zeros(L, bool)
        if hi > lo:
            mask[lo:hi] = True
        assert (after[b][mask] == 0).all(), b
        assert np.array_equal(after[b][~mask], before[b][~mask]), b


@pytest.mark.gpu
def test_gpu_after_spec_verify(sv):
    """The emitted counts of a verified batch drive the rollback (workload 2, ragged lengths)."""
    from workloads import make_workload
    w = make_workload(2)
    t = w.device_tensors()
    _, num, _ = sv.verify(t["target_logits"], t["draft_logits"], t["draft_tokens"], t["draft_len"],
                          t["temperature"], t["uniforms"])
    torch.cuda.synchronize()
    n = np.arange(w.B) * 3 + 5
    tl, dl = run_rollback(sv, n, w.draft_len, num.cpu().numpy(), None, w.G)
    o = oracle_verify(w.target_logits, w.draft_logits, w.draft_tokens, w.draft_len, w.temperature,
                      w.uniforms)
    want_t, want_d, _ = kv_rollback(n, w.draft_len, o.out_num_emitted, None, w.G)
    assert np.array_equal(tl, want_t) and np.array_equal(dl, want_d)


@pytest.mark.gpu
def test_gpu_rollback_argument_errors(sv):
    dev = torch.device("cuda")
    z = torch.zeros(4, dtype=torch.int32, device=dev)
    with pytest.raises(sv.SpecVerifyError) as ei:
        sv.spec_verify_kv_rollback(z, None, z, None, z, None,
                                   cache=torch.zeros((4, 3, 10), dtype=torch.uint8, device=dev),
                                   gamma_max=2)
    assert "MISALIGNED" in str(ei.value)     # 10-byte entries
