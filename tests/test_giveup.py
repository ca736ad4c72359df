"""The device-side failure detector: every wait of the streaming kernel is bounded, and a wait that
runs out sets the workspace status word, marks the rows the kernel was working on as errors and
ends the kernel, with the GPU context still usable.

The wait is made to run out without a fault: a test build of the library (compiled here, into a
temporary directory, never the library the package loads) has a small spin limit and a hook that
drops rank 0's exchange pushes, so every exchange waits for bytes that nothing sends.
"""
import ctypes
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_55_gb300 as m
    m.build_library()
    return m


@pytest.fixture(scope="module")
def starved_lib(tmp_path_factory):
    """The library built with a 4096-poll spin limit and rank 0's exchange pushes dropped."""
    from speculative_decoding_verification_55_gb300.build import build_library
    out = tmp_path_factory.mktemp("giveup") / "libspecverify_giveup.so"
    build_library(force=True, out=out,
                  extra_flags=["-DSV_SPIN_LIMIT=4096", "-DSV_TEST_DROP_RANK0_PUSHES"])
    L = ctypes.CDLL(str(out))
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    L.spec_verify_ex.argtypes = [vp] * 11 + [i32] * 4 + [vp, ctypes.c_size_t, vp]
    L.spec_verify_ex.restype = ctypes.c_int
    L.spec_verify_workspace_size.argtypes = [i32] * 4
    L.spec_verify_workspace_size.restype = ctypes.c_size_t
    L.spec_verify_workspace_status.argtypes = [vp, i32, i32, ctypes.POINTER(ctypes.c_int32), vp]
    L.spec_verify_workspace_status.restype = ctypes.c_int
    return L


def inputs(B, G, V, seed=0):
    rng = np.random.default_rng(seed)
    dev = torch.device("cuda")
    zt = torch.from_numpy(rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)).to(dev)
    zd = torch.from_numpy(rng.normal(0, 2, (B, G, V)).astype(np.float32)).to(dev)
    tok = torch.from_numpy(rng.integers(0, V, (B, G)).astype(np.int32)).to(dev)
    T = torch.ones((B,), dtype=torch.float32, device=dev)
    u = torch.from_numpy(rng.random((B, G + 2), dtype=np.float32)).to(dev)
    return zt, zd, tok, T, u


def test_a_wait_that_runs_out_is_reported_and_the_context_survives(sv, starved_lib):
    B, G, V = 2, 1, 4096                       # 16 KB fp32 rows: four one-CTA clusters
    zt, zd, tok, T, u = inputs(B, G, V)
    dev = zt.device
    out_tok = torch.full((B, G + 1), -7, dtype=torch.int32, device=dev)
    out_num = torch.full((B,), -7, dtype=torch.int32, device=dev)
    out_a = torch.full((B, G), -7.0, dtype=torch.float32, device=dev)
    L = starved_lib
    need = L.spec_verify_workspace_size(B, G, V, sv.SV_DTYPE_F32)
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.monotonic()
    st = L.spec_verify_ex(zt.data_ptr(), zd.data_ptr(), tok.data_ptr(), None, T.data_ptr(),
                          u.data_ptr(), out_tok.data_ptr(), out_num.data_ptr(), out_a.data_ptr(),
                          None, None, B, G, V, sv.SV_DTYPE_F32, ws.data_ptr(), need, stream)
    assert st == 0
    torch.cuda.synchronize()                   # returns: every wait is bounded
    assert time.monotonic() - t0 < 60
    status = ctypes.c_int32(-1)
    assert L.spec_verify_workspace_status(ws.data_ptr(), B, G, ctypes.byref(status), stream) == 0
    assert status.value == 1                   # the timeout bit
    assert out_num.tolist() == [-1] * B        # every row the kernel was working on is marked
    assert (out_tok == -1).all() and (out_a == 0).all()

    # The context is still usable: the package's own library verifies the same batch correctly.
    from oracle.spec_verify_oracle import oracle_verify
    from _parity import compare
    got = sv.verify(zt, zd, tok, None, T, u, with_probs=True)
    torch.cuda.synchronize()
    o = oracle_verify(zt.cpu().numpy(), zd.cpu().numpy(), tok.cpu().numpy(), None,
                      T.cpu().numpy(), u.cpu().numpy(), diagnostics=True)
    rep = compare(o, *[g.cpu().numpy() for g in got], tok.cpu().numpy(), np.full(B, G))
    assert rep.ok(), str(rep)
