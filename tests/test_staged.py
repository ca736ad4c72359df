"""spec_verify_staged: host buffers in, only the logit rows the rule reads copied to the device
(target rows 0..gamma_b, and draft rows 0..gamma_b - 1 of sampled rows: [R] "Speculative decoding",
rayaq.ca ml-models -- Mechanics, One round, steps 3-5; The greedy case), the verification, the
outputs copied back. CPU tests: the byte count against a brute-force count, the staging size, and
argument errors returned before any CUDA call. GPU tests: the staged call gives exactly the outputs
of spec_verify on device tensors, with every padding byte of the staging buffer left as NaN."""
import ctypes

import numpy as np
import pytest

SV_OK, SV_ERR_NULL_POINTER, SV_ERR_BAD_SHAPE, SV_ERR_WORKSPACE_TOO_SMALL, SV_ERR_MISALIGNED = 0, 1, 2, 4, 5


@pytest.fixture(scope="module")
def m():
    import speculative_decoding_verification_55_gb300 as sv
    sv.build_library()
    return sv


def brute_force_h2d(draft_len, temperature, B, G, V, s):
    """Bytes of every row the rule reads, row by row, plus the small inputs."""
    n = B * G * 4 + (B * 4 if draft_len is not None else 0) + B * 4 + B * (G + 2) * 4
    for b in range(B):
        g = G if draft_len is None else int(draft_len[b])
        if not 0 <= g <= G:
            continue
        n += (g + 1) * V * s                       # target rows 0..g
        if temperature[b] != 0.0:
            n += g * V * s                         # draft rows 0..g-1
    return n


@pytest.mark.parametrize("B,G,V,dtype", [(1, 0, 7, 0), (5, 3, 256, 0), (64, 8, 1000, 1),
                                         (300, 4, 33, 1)])
def test_h2d_bytes_match_a_row_by_row_count(m, B, G, V, dtype):
    rng = np.random.default_rng(B + G + V)
    s = 2 if dtype == 1 else 4
    for trial in range(6):
        draft_len = rng.integers(-2, G + 3, B).astype(np.int32)      # some out of [0, G]
        if trial == 0:
            draft_len[:] = G                                          # every run merges
        temperature = rng.uniform(0.2, 2.0, B).astype(np.float32)
        temperature[rng.random(B) < 0.3] = 0.0                        # greedy rows
        temperature[rng.random(B) < 0.05] = np.nan                    # copied like sampled rows
        for dl in (draft_len, None):
            want = brute_force_h2d(dl, temperature, B, G, V, s)
            assert m.spec_verify_staged_h2d_bytes(dl, temperature, B, G, V, dtype) == want


def test_staging_size(m):
    assert m.spec_verify_staging_size(0, 4, 100, 0) == 0
    assert m.spec_verify_staging_size(4, -1, 100, 0) == 0
    assert m.spec_verify_staging_size(4, 4, 100, 7) == 0
    for B, G, V, dt in [(1, 0, 1, 0), (8, 4, 32000, 1), (1024, 8, 256000, 1)]:
        s = 2 if dt == 1 else 4
        n = m.spec_verify_staging_size(B, G, V, dt)
        parts = [B * (G + 1) * V * s, B * G * V * s, B * G * 4, B * 4, B * 4, B * (G + 2) * 4,
                 B * (G + 1) * 4, B * 4, B * G * 4]
        assert n % 256 == 0
        assert sum(parts) <= n <= sum(parts) + 256 * len(parts)


def test_argument_errors_before_any_copy(m):
    """Fake addresses that are never dereferenced: every status here comes from the host checks."""
    L = m.lib()
    B, G, V = 4, 2, 64
    host = ctypes.c_void_p(0x10000)
    T = np.ones(B, np.float32)
    n = ctypes.c_size_t(123)
    need = m.spec_verify_staging_size(B, G, V, 0)
    ws = m.spec_verify_workspace_size(B, G, V, 0)

    def call(staging, staging_bytes, h_temp=T.ctypes.data, V_=V, zt=host):
        return L.spec_verify_staged(zt, host, host, None, h_temp, host, host, host, host, B, G, V_,
                                    0, staging, staging_bytes, ctypes.c_void_p(0x20000), ws,
                                    ctypes.byref(n), None)

    assert call(None, need) == SV_ERR_NULL_POINTER
    assert call(ctypes.c_void_p(0x30000), need, zt=None) == SV_ERR_NULL_POINTER
    assert call(ctypes.c_void_p(0x30080), need) == SV_ERR_MISALIGNED
    assert call(ctypes.c_void_p(0x30000), need - 1) == SV_ERR_WORKSPACE_TOO_SMALL
    assert call(ctypes.c_void_p(0x30000), need, V_=0) == SV_ERR_BAD_SHAPE
    assert n.value == 123                           # nothing was enqueued


# ------------------------------------------------------------------------------------------------

torch = pytest.importorskip("torch")


def staged_vs_device(m, w, bad_rows=(), pinned=True):
    t = w.device_tensors("cuda")
    if bad_rows:
        dl = t["draft_len"].clone()
        for b in bad_rows:
            dl[b] = w.G + 1 if b % 2 else -1
        t["draft_len"] = dl
    host = {k: (v.cpu().pin_memory() if pinned else v.cpu().clone()) for k, v in t.items()}
    want = [o.cpu() for o in m.verify(t["target_logits"], t["draft_logits"], t["draft_tokens"],
                                      t["draft_len"], t["temperature"], t["uniforms"])]
    B, G, V = w.B, w.G, w.V
    dt = 1 if t["target_logits"].dtype == torch.bfloat16 else 0
    staging = torch.full((m.spec_verify_staging_size(B, G, V, dt),), 0xFF, dtype=torch.uint8,
                         device="cuda")           # NaN in every unread logit byte
    ws = torch.zeros(m.spec_verify_workspace_size(B, G, V, dt), dtype=torch.uint8, device="cuda")
    out = [torch.empty((B, G + 1), dtype=torch.int32).pin_memory(),
           torch.empty((B,), dtype=torch.int32).pin_memory(),
           torch.empty((B, G), dtype=torch.float32).pin_memory()]
    n = m.spec_verify_staged(host["target_logits"], host["draft_logits"], host["draft_tokens"],
                             host["draft_len"], host["temperature"], host["uniforms"], *out,
                             staging, ws)
    torch.cuda.synchronize()
    assert n == m.spec_verify_staged_h2d_bytes(host["draft_len"], host["temperature"], B, G, V, dt)
    assert n == brute_force_h2d(host["draft_len"].numpy(), host["temperature"].numpy(), B, G, V,
                                2 if dt else 4)
    for a, b in zip(out, want):
        assert torch.equal(a, b)
    for b in bad_rows:
        assert out[1][b] == -1
    return n


@pytest.mark.gpu
@pytest.mark.parametrize("key,pinned", [(1, True), (2, True), (2, False), (3, True), (4, True),
                                        (3, False)])
def test_gpu_staged_matches_device_call(m, key, pinned):
    """Page-locked host buffers take the zero-copy gather; pageable ones the per-run copies."""
    from workloads import make_workload
    w = make_workload(key, backend="numpy" if key <= 2 else "torch",
                      device=None if key <= 2 else "cuda")
    staged_vs_device(m, w, bad_rows=(0,) if key == 3 else (), pinned=pinned)


@pytest.mark.gpu
def test_gpu_staged_full_size_ragged_batch(m):
    """The benchmark's ragged batch: about 4.9 GB of the padded 8.9 GB is copied."""
    from workloads import make_workload
    w = make_workload(5, backend="torch", device="cuda")
    n = staged_vs_device(m, w)
    assert n < 0.6 * (w.B * (2 * w.G + 1) * w.V * 2)
