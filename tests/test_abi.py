"""The C-ABI library builds, loads, exports every function include/spec_verify.h declares, and rejects
bad arguments on the host before touching the GPU. CPU only: no compute call is made."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "spec_verify.h"


@pytest.fixture(scope="module")
def L():
    import speculative_decoding_verification_55_gb300 as m
    m.build_library()
    return m.lib()


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_verify\w*)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ("spec_verify", "spec_verify_ex", "spec_verify_workspace_size",
              "spec_verify_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    import speculative_decoding_verification_55_gb300 as m
    for name in declared_functions():
        assert callable(getattr(m, name)), name


def test_version_and_status_strings(L):
    import speculative_decoding_verification_55_gb300 as m
    assert m.spec_verify_version() == 1
    for code in range(8):
        s = m.spec_verify_status_string(code)
        assert s.startswith("SV_")
    assert "unknown" in m.spec_verify_status_string(99)


def test_workspace_size(L):
    import speculative_decoding_verification_55_gb300 as m
    for B, G in ((1, 0), (1, 4), (8, 4), (1024, 8), (7, 64)):
        n = m.spec_verify_workspace_size(B, G, 32000, 1)
        assert n % 256 == 0 and n >= 8 * B * (G + 1) + 4 * B
    for B, G in ((1, 0), (8, 4), (1024, 8)):
        n = m.spec_verify_workspace_size(B, G, 32000, 1)
        f = m.spec_verify_filtered_workspace_size(B, G, 32000, 1)
        assert f % 256 == 0 and f >= n + 128 * 8 * B * (2 * G + 1)
    assert m.spec_verify_filtered_workspace_size(0, 4, 100, 0) == 0
    assert m.spec_verify_workspace_size(0, 4, 100, 0) == 0
    assert m.spec_verify_workspace_size(2, 65, 100, 0) == 0
    assert m.spec_verify_workspace_size(2, -1, 100, 0) == 0
    assert m.spec_verify_workspace_size(2, 4, 0, 0) == 0
    assert m.spec_verify_workspace_size(2, 4, 100, 7) == 0


FAKE = 0x7f0000000000   # never dereferenced: every case below fails validation first


def call(L, **kw):
    B, G, V, dtype = kw.get("B", 2), kw.get("G", 3), kw.get("V", 256), kw.get("dtype", 1)
    args = dict(zt=FAKE, zd=FAKE + 4096, tok=FAKE + 8192, dl=FAKE + 12288, T=FAKE + 16384,
                u=FAKE + 20480, ot=FAKE + 24576, on=FAKE + 28672, oa=FAKE + 32768,
                ws=FAKE + 65536, wsb=1 << 20)
    args.update({k: v for k, v in kw.items() if k in args})
    return L.spec_verify(args["zt"], args["zd"], args["tok"], args["dl"], args["T"], args["u"],
                         args["ot"], args["on"], args["oa"], B, G, V, dtype, args["ws"],
                         args["wsb"], None)


def test_argument_errors_are_host_side(L):
    assert call(L, dtype=5) == 3                      # SV_ERR_BAD_DTYPE
    assert call(L, B=0) == 2                          # SV_ERR_BAD_SHAPE
    assert call(L, G=65) == 2
    assert call(L, V=0) == 2
    assert call(L, zt=None) == 1                      # SV_ERR_NULL_POINTER
    assert call(L, T=None) == 1
    assert call(L, u=None) == 1
    assert call(L, ot=None) == 1
    assert call(L, on=None) == 1
    assert call(L, zd=None) == 1                      # needed when G > 0
    assert call(L, zt=FAKE + 1) == 5                  # SV_ERR_MISALIGNED (bf16 needs 2 B)
    assert call(L, dtype=0, zt=FAKE + 2) == 5         # fp32 needs 4 B
    assert call(L, ws=FAKE + 65544) == 5              # workspace needs 16 B
    assert call(L, ws=None) == 4                      # SV_ERR_WORKSPACE_TOO_SMALL
    assert call(L, wsb=16) == 4
    # Rows whose byte length is not a multiple of 16 take the element path, which holds at most
    # 16 * 512 * 32 logits per row; 16-byte rows stream, up to 1048576 bf16 or 311296 fp32 logits.
    assert call(L, V=262145) == 2
    assert call(L, dtype=0, V=262147) == 2
    assert call(L, V=1048576 + 8) == 2
    assert call(L, dtype=0, V=311296 + 4) == 2


def call_filtered(L, **kw):
    B, G, V, dtype = kw.get("B", 2), kw.get("G", 3), kw.get("V", 256), kw.get("dtype", 1)
    args = dict(zt=FAKE, zd=FAKE + 4096, tok=FAKE + 8192, dl=FAKE + 12288, T=FAKE + 16384,
                tk=FAKE + 17408, tp=FAKE + 18432, u=FAKE + 20480, ot=FAKE + 24576,
                on=FAKE + 28672, oa=FAKE + 32768, ws=FAKE + 65536, wsb=1 << 20)
    args.update({k: v for k, v in kw.items() if k in args})
    return L.spec_verify_filtered(args["zt"], args["zd"], args["tok"], args["dl"], args["T"],
                                  args["tk"], args["tp"], args["u"], args["ot"], args["on"],
                                  args["oa"], None, None, B, G, V, dtype, args["ws"], args["wsb"],
                                  None)


def test_filtered_argument_errors_are_host_side(L):
    """spec_verify_filtered checks everything before it touches the device (16-byte rows only)."""
    assert call_filtered(L, dtype=5) == 3             # SV_ERR_BAD_DTYPE
    assert call_filtered(L, B=0) == 2                 # SV_ERR_BAD_SHAPE
    assert call_filtered(L, G=65) == 2
    assert call_filtered(L, zt=None) == 1             # SV_ERR_NULL_POINTER
    assert call_filtered(L, zd=None) == 1
    assert call_filtered(L, tk=FAKE + 17409) == 5     # SV_ERR_MISALIGNED: top_k needs 4 B
    assert call_filtered(L, tp=FAKE + 18434) == 5     # top_p needs 4 B
    assert call_filtered(L, zt=FAKE + 8) == 5         # logit bases need 16 B here
    assert call_filtered(L, V=257) == 2               # 514-byte rows: not a multiple of 16
    assert call_filtered(L, ws=None) == 4             # SV_ERR_WORKSPACE_TOO_SMALL
    assert call_filtered(L, V=16 * 65536 + 8) == 2    # more than 16 chunks of the row buffer


def test_tree_onehot_rollback_argument_errors_are_host_side(L):
    """The tree, one-hot and rollback entry points reject bad arguments before any device call."""
    def tree(**kw):
        a = dict(zt=FAKE, tok=FAKE + 4096, par=FAKE + 8192, size=None, path=FAKE + 12288,
                 plen=FAKE + 16384, otok=FAKE + 20480, pred=None, ws=FAKE + 65536, wsb=1 << 20,
                 B=2, N=7, V=256, dtype=1)
        a.update(kw)
        return L.spec_verify_tree_greedy(a["zt"], a["tok"], a["par"], a["size"], a["path"],
                                         a["plen"], a["otok"], a["pred"], a["B"], a["N"], a["V"],
                                         a["dtype"], a["ws"], a["wsb"], None)

    assert tree(dtype=5) == 3
    assert tree(N=0) == 2 and tree(N=66) == 2          # N - 1 drafted levels at most SV_MAX_GAMMA
    assert tree(zt=None) == 1 and tree(par=None) == 1 and tree(path=None) == 1
    assert tree(tok=FAKE + 4097) == 5
    assert tree(ws=None) == 4
    assert tree(V=257) == 2                            # 514-byte rows: streaming kernel only
    assert tree(zt=FAKE + 8) == 5                      # row bases need 16 B

    def onehot(**kw):
        a = dict(zt=FAKE, tok=FAKE + 8192, dl=FAKE + 12288, T=FAKE + 16384, u=FAKE + 20480,
                 ot=FAKE + 24576, on=FAKE + 28672, oa=FAKE + 32768, ws=FAKE + 65536, wsb=1 << 20,
                 B=2, G=3, V=256, dtype=1)
        a.update(kw)
        return L.spec_verify_onehot(a["zt"], a["tok"], a["dl"], a["T"], a["u"], a["ot"], a["on"],
                                    a["oa"], None, None, a["B"], a["G"], a["V"], a["dtype"], a["ws"],
                                    a["wsb"], None)

    assert onehot(dtype=5) == 3
    assert onehot(B=0) == 2
    assert onehot(tok=None) == 1                       # drafted tokens are needed when G > 0
    assert onehot(T=FAKE + 16385) == 5
    assert onehot(ws=None) == 4
    assert onehot(V=257) == 2                          # one-hot drafts: streaming kernel only
    assert onehot(zt=FAKE + 8) == 5

    def rollback(**kw):
        a = dict(pre=FAKE, dl=None, num=FAKE + 4096, din=None, tout=FAKE + 8192, dout=None,
                 cache=None, stride=0, eb=0, ne=0, B=2, G=3)
        a.update(kw)
        return L.spec_verify_kv_rollback(a["pre"], a["dl"], a["num"], a["din"], a["tout"],
                                         a["dout"], a["cache"], a["stride"], a["eb"], a["ne"],
                                         a["B"], a["G"], None)

    assert rollback(B=0) == 2 and rollback(G=65) == 2
    assert rollback(pre=None) == 1 and rollback(num=None) == 1 and rollback(tout=None) == 1
    assert rollback(num=FAKE + 4098) == 5
    assert rollback(cache=FAKE + 65536, eb=0, ne=4, stride=1024) == 2      # no entry size
    assert rollback(cache=FAKE + 65536, eb=256, ne=8, stride=1024) == 2    # stride < 8 entries
    assert rollback(cache=FAKE + 65536, eb=24, ne=4, stride=1024) == 5     # entries of 16 B
    assert rollback(cache=FAKE + 65544, eb=256, ne=4, stride=1024) == 5    # cache base 16 B


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import speculative_decoding_verification_55_gb300._binding as b
    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "LIB_PATH", tmp_path / "missing.so")
    with pytest.raises(RuntimeError, match="missing"):
        b.lib()
