"""spec_verify_noalloc: the entry point for callers that cannot allocate device memory (engines that
plan all device memory at start-up and forbid allocation while serving, hosts that cannot pay for
cudaMalloc's synchronisation, plugin interfaces that receive only input and output buffers). It
keeps the kernels' scratch in the library's static device array instead of a caller workspace.

This file is collected last on purpose, so that a run stopping at its first failure has already
run every other test. It must pass alone in a fresh process and after the other tests.
"""
import numpy as np
import pytest

from workloads import make_workload

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 1e-5


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_55_gb300 as m
    m.build_library()
    return m


def outputs(t, B, G):
    dev = t["target_logits"].device
    return (torch.full((B, G + 1), -7, dtype=torch.int32, device=dev),
            torch.full((B,), -7, dtype=torch.int32, device=dev),
            torch.full((B, G), -7.0, dtype=torch.float32, device=dev),
            torch.full((B, G), -7.0, dtype=torch.float32, device=dev),
            torch.full((B, G), -7.0, dtype=torch.float32, device=dev))


def test_noalloc_matches_workspace_entry_point_and_oracle_twice(sv):
    """Two calls in a row (different batch shapes, so the shared scratch is reused with a new
    layout) give the same outputs as spec_verify_ex with a caller workspace, and match the fp64
    oracle under the margin rule of the parity tests."""
    from _parity import compare
    from oracle.spec_verify_oracle import oracle_verify
    for key in (2, 3):
        w = make_workload(key)
        t = w.device_tensors()
        B, G = w.B, w.G
        ref = sv.verify(t["target_logits"], t["draft_logits"], t["draft_tokens"], t["draft_len"],
                        t["temperature"], t["uniforms"], with_probs=True)
        out = outputs(t, B, G)
        sv.spec_verify_noalloc(t["target_logits"], t["draft_logits"], t["draft_tokens"],
                               t["draft_len"], t["temperature"], t["uniforms"], *out)
        torch.cuda.synchronize()
        assert torch.equal(out[0], ref[0]) and torch.equal(out[1], ref[1]), key
        for a, b in zip(out[2:], ref[2:]):
            assert float((a - b).abs().max()) <= TOL, key
        assert int(out[1].min()) >= 1
        o = oracle_verify(w.target_logits, w.draft_logits, w.draft_tokens, w.draft_len,
                          w.temperature, w.uniforms, diagnostics=True)
        rep = compare(o, *[a.cpu().numpy() for a in out], w.draft_tokens, w.draft_len)
        assert rep.ok(), f"workload {key}: {rep}"


def test_noalloc_rejected_call_enqueues_nothing(sv):
    """A call rejected for a bad argument returns the status spec_verify_ex returns and writes no
    output (nothing was enqueued)."""
    w = make_workload(2)
    t = w.device_tensors()
    B, G = w.B, w.G
    ws = sv.workspace_for(B, G, w.V, sv.SV_DTYPE_BF16, t["target_logits"].device)
    raw = sv.lib()
    out = outputs(t, B, G)
    zt = t["target_logits"]
    args = [zt.data_ptr() + 1, t["draft_logits"].data_ptr(), t["draft_tokens"].data_ptr(),
            t["draft_len"].data_ptr(), t["temperature"].data_ptr(), t["uniforms"].data_ptr()] + \
        [o.data_ptr() for o in out]
    tail = [B, G, w.V, sv.SV_DTYPE_BF16]
    stream = torch.cuda.current_stream().cuda_stream
    cases = {"misaligned": args, "null": [None] + args[1:]}
    for name, a in cases.items():
        st_ex = raw.spec_verify_ex(*a, *tail, ws.data_ptr(), ws.numel(), stream)
        st_na = raw.spec_verify_noalloc(*a, *tail, stream)
        assert st_na == st_ex != 0, (name, st_na, st_ex)
    torch.cuda.synchronize()
    assert int((out[1] == -7).sum()) == B and int((out[0] == -7).sum()) == out[0].numel()


def test_noalloc_rejects_sizes_beyond_its_scratch(sv):
    B, G, V = 70000, 1, 8
    assert sv.spec_verify_workspace_size(B, G, V, sv.SV_DTYPE_F32) > sv.SV_NOALLOC_SCRATCH_BYTES
    dev = torch.device("cuda")
    zt = torch.zeros((B, G + 1, V), dtype=torch.float32, device=dev)
    zd = torch.zeros((B, G, V), dtype=torch.float32, device=dev)
    tok = torch.zeros((B, G), dtype=torch.int32, device=dev)
    T = torch.ones((B,), dtype=torch.float32, device=dev)
    u = torch.zeros((B, G + 2), dtype=torch.float32, device=dev)
    out = outputs(dict(target_logits=zt), B, G)
    with pytest.raises(sv.SpecVerifyError) as ei:
        sv.spec_verify_noalloc(zt, zd, tok, None, T, u, *out)
    assert ei.value.status == sv.SV_ERR_SCRATCH_TOO_SMALL
    assert "static scratch" in str(ei.value)
    assert int((out[1] == -7).sum()) == B          # nothing was launched
