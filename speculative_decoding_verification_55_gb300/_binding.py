"""ctypes binding of libspecverify.so: the C ABI in include/spec_verify.h under the same names.

Argument marshalling only: every step of the verification runs in the library's CUDA kernels.
Torch tensors supply device memory and the stream. There is no CPU fallback: if the library is not
built, importing the functions raises.
"""
from __future__ import annotations

import ctypes
import threading

from .build import LIB_PATH

SV_OK = 0
SV_DTYPE_F32 = 0
SV_DTYPE_BF16 = 1
SV_MAX_GAMMA = 64

STATUS_NAMES = {
    0: "SV_OK", 1: "SV_ERR_NULL_POINTER", 2: "SV_ERR_BAD_SHAPE", 3: "SV_ERR_BAD_DTYPE",
    4: "SV_ERR_WORKSPACE_TOO_SMALL", 5: "SV_ERR_MISALIGNED", 6: "SV_ERR_CUDA",
    7: "SV_ERR_UNSUPPORTED_DEVICE", 8: "SV_ERR_SCRATCH_TOO_SMALL",
}
SV_ERR_SCRATCH_TOO_SMALL = 8
SV_NOALLOC_SCRATCH_BYTES = 1 << 20

EXPORTED = ("spec_verify", "spec_verify_ex", "spec_verify_noalloc", "spec_verify_onehot",
            "spec_verify_filtered", "spec_verify_filter_thresholds", "spec_verify_tree_greedy",
            "spec_verify_kv_rollback",
            "spec_verify_workspace_size", "spec_verify_filtered_workspace_size",
            "spec_verify_workspace_status", "spec_verify_status_string",
            "spec_verify_version")

_lib = None
_lock = threading.Lock()


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, where: str = "spec_verify"):
        self.status = status
        super().__init__(f"{where} returned {status} ({spec_verify_status_string(status)})")


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not LIB_PATH.exists():
                raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                                   "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(str(LIB_PATH))
            vp, i32, f32p, i32p = ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p
            common = [vp, vp, i32p, i32p, f32p, f32p, i32p, i32p, f32p]
            tail = [i32, i32, i32, i32, vp, ctypes.c_size_t, vp]
            L.spec_verify.argtypes = common + tail
            L.spec_verify.restype = ctypes.c_int
            L.spec_verify_ex.argtypes = common + [f32p, f32p] + tail
            L.spec_verify_ex.restype = ctypes.c_int
            L.spec_verify_noalloc.argtypes = common + [f32p, f32p, i32, i32, i32, i32, vp]
            L.spec_verify_noalloc.restype = ctypes.c_int
            L.spec_verify_onehot.argtypes = [vp, i32p, i32p, f32p, f32p, i32p, i32p, f32p, f32p, f32p] + tail
            L.spec_verify_onehot.restype = ctypes.c_int
            L.spec_verify_filtered.argtypes = [vp, vp, i32p, i32p, f32p, i32p, f32p, f32p, i32p, i32p,
                                               f32p, f32p, f32p] + tail
            L.spec_verify_filtered.restype = ctypes.c_int
            L.spec_verify_filter_thresholds.argtypes = [vp, vp, i32p, f32p, i32p, f32p, f32p, i32, i32,
                                                        i32, i32, vp]
            L.spec_verify_filter_thresholds.restype = ctypes.c_int
            L.spec_verify_tree_greedy.argtypes = [vp, i32p, i32p, i32p, i32p, i32p, i32p, i32p] + tail
            L.spec_verify_tree_greedy.restype = ctypes.c_int
            L.spec_verify_kv_rollback.argtypes = [i32p, i32p, i32p, i32p, i32p, i32p, vp, ctypes.c_int64,
                                                  i32, i32, i32, i32, vp]
            L.spec_verify_kv_rollback.restype = ctypes.c_int
            L.spec_verify_workspace_size.argtypes = [i32, i32, i32, i32]
            L.spec_verify_workspace_size.restype = ctypes.c_size_t
            L.spec_verify_filtered_workspace_size.argtypes = [i32, i32, i32, i32]
            L.spec_verify_filtered_workspace_size.restype = ctypes.c_size_t
            L.spec_verify_workspace_status.argtypes = [vp, i32, i32, ctypes.POINTER(ctypes.c_int32), vp]
            L.spec_verify_workspace_status.restype = ctypes.c_int
            L.spec_verify_status_string.argtypes = [ctypes.c_int]
            L.spec_verify_status_string.restype = ctypes.c_char_p
            L.spec_verify_version.argtypes = []
            L.spec_verify_version.restype = ctypes.c_int
            L.spec_verify_staging_size.argtypes = [i32, i32, i32, i32]
            L.spec_verify_staging_size.restype = ctypes.c_size_t
            L.spec_verify_staged_h2d_bytes.argtypes = [vp, vp, i32, i32, i32, i32]
            L.spec_verify_staged_h2d_bytes.restype = ctypes.c_size_t
            L.spec_verify_staged.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                             vp, ctypes.c_size_t, vp, ctypes.c_size_t,
                                             ctypes.POINTER(ctypes.c_size_t), vp]
            L.spec_verify_staged.restype = ctypes.c_int
            _lib = L
    return _lib


def spec_verify_workspace_size(B: int, gamma_max: int, V: int, dtype: int) -> int:
    return int(lib().spec_verify_workspace_size(B, gamma_max, V, dtype))


def spec_verify_filtered_workspace_size(B: int, gamma_max: int, V: int, dtype: int) -> int:
    return int(lib().spec_verify_filtered_workspace_size(B, gamma_max, V, dtype))


def spec_verify_status_string(status: int) -> str:
    return lib().spec_verify_status_string(int(status)).decode()


def spec_verify_workspace_status(workspace, B: int, gamma_max: int, stream=None) -> int:
    """The workspace's sticky status word (0 = every call completed its protocol)."""
    out = ctypes.c_int32(0)
    with _on(workspace.device):
        st = lib().spec_verify_workspace_status(_ptr(workspace), B, gamma_max, ctypes.byref(out),
                                                _stream_handle(stream, workspace.device))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_workspace_status")
    return int(out.value)


def spec_verify_version() -> int:
    return int(lib().spec_verify_version())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return SV_DTYPE_BF16
    if t.dtype == torch.float32:
        return SV_DTYPE_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _check(t, name, dtype=None, shape=None, device=None):
    if t is None:
        return
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


def _on(device):
    """The CUDA device of the call's buffers made current for the C call: the library launches on
    (and, for spec_verify_noalloc, takes the scratch address of) the current device."""
    import contextlib
    import torch
    if device is None or device.type != "cuda":
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def spec_verify_ex(target_logits, draft_logits, draft_tokens, draft_len, temperature, uniforms,
                   out_tokens, out_num_emitted, out_alpha, out_p_draft, out_q_draft,
                   workspace, stream=None) -> None:
    """Calls the C ABI spec_verify_ex on torch tensors (shapes from target_logits [B, G+1, V]).
    Raises SpecVerifyError on a nonzero status."""
    import torch
    B, G1, V = target_logits.shape
    G = G1 - 1
    dev = target_logits.device
    _check(target_logits, "target_logits", device=dev)
    _check(draft_logits, "draft_logits", dtype=target_logits.dtype, shape=(B, G, V), device=dev)
    _check(draft_tokens, "draft_tokens", torch.int32, (B, G), dev)
    _check(draft_len, "draft_len", torch.int32, (B,), dev)
    _check(temperature, "temperature", torch.float32, (B,), dev)
    _check(uniforms, "uniforms", torch.float32, (B, G + 2), dev)
    _check(out_tokens, "out_tokens", torch.int32, (B, G + 1), dev)
    _check(out_num_emitted, "out_num_emitted", torch.int32, (B,), dev)
    for name, t in (("out_alpha", out_alpha), ("out_p_draft", out_p_draft),
                    ("out_q_draft", out_q_draft)):
        _check(t, name, torch.float32, (B, G), dev)
    _check(workspace, "workspace", device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    with _on(dev):
        st = lib().spec_verify_ex(
            _ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), _ptr(draft_len),
            _ptr(temperature), _ptr(uniforms), _ptr(out_tokens), _ptr(out_num_emitted),
            _ptr(out_alpha), _ptr(out_p_draft), _ptr(out_q_draft),
            B, G, V, _dtype_code(target_logits), _ptr(workspace), ws_bytes,
            _stream_handle(stream, dev))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_ex")


def spec_verify_staging_size(B: int, gamma_max: int, V: int, dtype: int) -> int:
    return int(lib().spec_verify_staging_size(B, gamma_max, V, dtype))


def _host_ptr(a):
    """Address of a host buffer: a CPU torch tensor or a contiguous numpy array (None -> NULL)."""
    if a is None:
        return None
    if hasattr(a, "data_ptr"):
        if a.is_cuda:
            raise ValueError("expected a host (CPU) buffer")
        return a.data_ptr()
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("host arrays must be contiguous")
    return a.ctypes.data


def spec_verify_staged_h2d_bytes(draft_len, temperature, B: int, gamma_max: int, V: int,
                                 dtype: int) -> int:
    """Host-to-device bytes spec_verify_staged enqueues for these host draft lengths (int32, or
    None) and temperatures (float32)."""
    return int(lib().spec_verify_staged_h2d_bytes(_host_ptr(draft_len), _host_ptr(temperature),
                                                  B, gamma_max, V, dtype))


def spec_verify_staged(target_logits, draft_logits, draft_tokens, draft_len, temperature, uniforms,
                       out_tokens, out_num_emitted, out_alpha, staging, workspace,
                       stream=None) -> int:
    """Calls the C ABI spec_verify_staged: host (CPU, ideally pinned) torch tensors in and out,
    device staging and workspace buffers. Returns the host-to-device bytes enqueued."""
    import torch
    B, G1, V = target_logits.shape
    G = G1 - 1
    cpu = torch.device("cpu")
    _check(target_logits, "target_logits", device=cpu)
    _check(draft_logits, "draft_logits", dtype=target_logits.dtype, shape=(B, G, V), device=cpu)
    _check(draft_tokens, "draft_tokens", torch.int32, (B, G), cpu)
    _check(draft_len, "draft_len", torch.int32, (B,), cpu)
    _check(temperature, "temperature", torch.float32, (B,), cpu)
    _check(uniforms, "uniforms", torch.float32, (B, G + 2), cpu)
    _check(out_tokens, "out_tokens", torch.int32, (B, G + 1), cpu)
    _check(out_num_emitted, "out_num_emitted", torch.int32, (B,), cpu)
    _check(out_alpha, "out_alpha", torch.float32, (B, G), cpu)
    dev = staging.device
    _check(workspace, "workspace", device=dev)
    n = ctypes.c_size_t(0)
    with _on(dev):
        st = lib().spec_verify_staged(
            _host_ptr(target_logits), _host_ptr(draft_logits), _host_ptr(draft_tokens),
            _host_ptr(draft_len), _host_ptr(temperature), _host_ptr(uniforms), _host_ptr(out_tokens),
            _host_ptr(out_num_emitted), _host_ptr(out_alpha), B, G, V, _dtype_code(target_logits),
            _ptr(staging), staging.numel() * staging.element_size(), _ptr(workspace),
            workspace.numel() * workspace.element_size(), ctypes.byref(n), _stream_handle(stream, dev))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_staged")
    return int(n.value)


_staging_cache = {}


def verify_staged(target_logits, draft_logits, draft_tokens, draft_len, temperature, uniforms,
                  device=None, stream=None):
    """spec_verify_staged with pinned host outputs and a cached device staging buffer and
    workspace. Returns (out_tokens, out_num_emitted, out_alpha, h2d_bytes); the outputs are valid
    once the stream has been synchronised."""
    import torch
    B, G1, V = target_logits.shape
    G = G1 - 1
    device = torch.device(device or "cuda")
    dt = _dtype_code(target_logits)
    key = (str(device), _stream_handle(stream, device), B, G, V, dt)
    if key not in _staging_cache:
        _staging_cache[key] = torch.empty(spec_verify_staging_size(B, G, V, dt), dtype=torch.uint8,
                                          device=device)
    ws = workspace_for(B, G, V, dt, device, stream)
    out_tokens = torch.empty((B, G1), dtype=torch.int32).pin_memory()
    out_num = torch.empty((B,), dtype=torch.int32).pin_memory()
    out_alpha = torch.empty((B, G), dtype=torch.float32).pin_memory()
    n = spec_verify_staged(target_logits, draft_logits, draft_tokens, draft_len, temperature,
                           uniforms, out_tokens, out_num, out_alpha, _staging_cache[key], ws,
                           stream)
    return out_tokens, out_num, out_alpha, n


def spec_verify_noalloc(target_logits, draft_logits, draft_tokens, draft_len, temperature,
                        uniforms, out_tokens, out_num_emitted, out_alpha, out_p_draft=None,
                        out_q_draft=None, stream=None) -> None:
    """Calls the C ABI spec_verify_noalloc: like spec_verify_ex, with the library's static device
    scratch instead of a workspace (for callers that cannot allocate). Raises SpecVerifyError on a
    nonzero status, e.g. SV_ERR_SCRATCH_TOO_SMALL for sizes beyond SV_NOALLOC_SCRATCH_BYTES."""
    import torch
    B, G1, V = target_logits.shape
    G = G1 - 1
    dev = target_logits.device
    _check(target_logits, "target_logits", device=dev)
    _check(draft_logits, "draft_logits", dtype=target_logits.dtype, shape=(B, G, V), device=dev)
    _check(draft_tokens, "draft_tokens", torch.int32, (B, G), dev)
    _check(draft_len, "draft_len", torch.int32, (B,), dev)
    _check(temperature, "temperature", torch.float32, (B,), dev)
    _check(uniforms, "uniforms", torch.float32, (B, G + 2), dev)
    _check(out_tokens, "out_tokens", torch.int32, (B, G + 1), dev)
    _check(out_num_emitted, "out_num_emitted", torch.int32, (B,), dev)
    for name, t in (("out_alpha", out_alpha), ("out_p_draft", out_p_draft),
                    ("out_q_draft", out_q_draft)):
        _check(t, name, torch.float32, (B, G), dev)
    with _on(dev):
        st = lib().spec_verify_noalloc(
            _ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), _ptr(draft_len),
            _ptr(temperature), _ptr(uniforms), _ptr(out_tokens), _ptr(out_num_emitted),
            _ptr(out_alpha), _ptr(out_p_draft), _ptr(out_q_draft),
            B, G, V, _dtype_code(target_logits), _stream_handle(stream, dev))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_noalloc")


def spec_verify_onehot(target_logits, draft_tokens, draft_len, temperature, uniforms, out_tokens,
                       out_num_emitted, out_alpha, out_p_draft, out_q_draft, workspace,
                       stream=None) -> None:
    """Calls the C ABI spec_verify_onehot (one-hot drafts, no draft logits) on torch tensors.
    Raises SpecVerifyError on a nonzero status."""
    import torch
    B, G1, V = target_logits.shape
    G = G1 - 1
    dev = target_logits.device
    _check(target_logits, "target_logits", device=dev)
    _check(draft_tokens, "draft_tokens", torch.int32, (B, G), dev)
    _check(draft_len, "draft_len", torch.int32, (B,), dev)
    _check(temperature, "temperature", torch.float32, (B,), dev)
    _check(uniforms, "uniforms", torch.float32, (B, G + 2), dev)
    _check(out_tokens, "out_tokens", torch.int32, (B, G + 1), dev)
    _check(out_num_emitted, "out_num_emitted", torch.int32, (B,), dev)
    for name, t in (("out_alpha", out_alpha), ("out_p_draft", out_p_draft),
                    ("out_q_draft", out_q_draft)):
        _check(t, name, torch.float32, (B, G), dev)
    _check(workspace, "workspace", device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    with _on(dev):
        st = lib().spec_verify_onehot(
            _ptr(target_logits), _ptr(draft_tokens), _ptr(draft_len), _ptr(temperature),
            _ptr(uniforms), _ptr(out_tokens), _ptr(out_num_emitted), _ptr(out_alpha),
            _ptr(out_p_draft), _ptr(out_q_draft), B, G, V, _dtype_code(target_logits),
            _ptr(workspace), ws_bytes, _stream_handle(stream, dev))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_onehot")


def spec_verify_filtered(target_logits, draft_logits, draft_tokens, draft_len, temperature, top_k,
                         top_p, uniforms, out_tokens, out_num_emitted, out_alpha, out_p_draft,
                         out_q_draft, workspace, stream=None) -> None:
    """Calls the C ABI spec_verify_filtered (per-row top-k / top-p applied to p and q before the
    test) on torch tensors; top_k [B] int32 and top_p [B] float32 may be None (off).
    Raises SpecVerifyError on a nonzero status."""
    import torch
    B, G1, V = target_logits.shape
    G = G1 - 1
    dev = target_logits.device
    _check(target_logits, "target_logits", device=dev)
    _check(draft_logits, "draft_logits", dtype=target_logits.dtype, shape=(B, G, V), device=dev)
    _check(draft_tokens, "draft_tokens", torch.int32, (B, G), dev)
    _check(draft_len, "draft_len", torch.int32, (B,), dev)
    _check(temperature, "temperature", torch.float32, (B,), dev)
    _check(top_k, "top_k", torch.int32, (B,), dev)
    _check(top_p, "top_p", torch.float32, (B,), dev)
    _check(uniforms, "uniforms", torch.float32, (B, G + 2), dev)
    _check(out_tokens, "out_tokens", torch.int32, (B, G + 1), dev)
    _check(out_num_emitted, "out_num_emitted", torch.int32, (B,), dev)
    for name, t in (("out_alpha", out_alpha), ("out_p_draft", out_p_draft),
                    ("out_q_draft", out_q_draft)):
        _check(t, name, torch.float32, (B, G), dev)
    _check(workspace, "workspace", device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    with _on(dev):
        st = lib().spec_verify_filtered(
            _ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), _ptr(draft_len),
            _ptr(temperature), _ptr(top_k), _ptr(top_p), _ptr(uniforms), _ptr(out_tokens),
            _ptr(out_num_emitted), _ptr(out_alpha), _ptr(out_p_draft), _ptr(out_q_draft),
            B, G, V, _dtype_code(target_logits), _ptr(workspace), ws_bytes,
            _stream_handle(stream, dev))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_filtered")


def spec_verify_filter_thresholds(target_logits, draft_logits, draft_len, temperature, top_k, top_p,
                                  out_thresholds, stream=None) -> None:
    """Calls the C ABI spec_verify_filter_thresholds: per logit row the smallest logit top-k /
    top-p keep (-inf where nothing is filtered) into out_thresholds [B * (2G + 1)] float32.
    Raises SpecVerifyError on a nonzero status."""
    import torch
    B, G1, V = target_logits.shape
    G = G1 - 1
    dev = target_logits.device
    _check(target_logits, "target_logits", device=dev)
    _check(draft_logits, "draft_logits", dtype=target_logits.dtype, shape=(B, G, V), device=dev)
    _check(draft_len, "draft_len", torch.int32, (B,), dev)
    _check(temperature, "temperature", torch.float32, (B,), dev)
    _check(top_k, "top_k", torch.int32, (B,), dev)
    _check(top_p, "top_p", torch.float32, (B,), dev)
    _check(out_thresholds, "out_thresholds", torch.float32, (B * (2 * G + 1),), dev)
    with _on(dev):
        st = lib().spec_verify_filter_thresholds(
            _ptr(target_logits), _ptr(draft_logits), _ptr(draft_len), _ptr(temperature),
            _ptr(top_k), _ptr(top_p), _ptr(out_thresholds), B, G, V, _dtype_code(target_logits),
            _stream_handle(stream, dev))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_filter_thresholds")


def spec_verify_tree_greedy(target_logits, tree_tokens, tree_parents, tree_size, out_path,
                            out_path_len, out_tokens, out_pred, workspace, stream=None) -> None:
    """Calls the C ABI spec_verify_tree_greedy (greedy verification of candidate trees) on torch
    tensors: target_logits [B, N, V]. Raises SpecVerifyError on a nonzero status."""
    import torch
    B, N, V = target_logits.shape
    dev = target_logits.device
    _check(target_logits, "target_logits", device=dev)
    _check(tree_tokens, "tree_tokens", torch.int32, (B, N), dev)
    _check(tree_parents, "tree_parents", torch.int32, (B, N), dev)
    _check(tree_size, "tree_size", torch.int32, (B,), dev)
    _check(out_path, "out_path", torch.int32, (B, N), dev)
    _check(out_path_len, "out_path_len", torch.int32, (B,), dev)
    _check(out_tokens, "out_tokens", torch.int32, (B, N + 1), dev)
    _check(out_pred, "out_pred", torch.int32, (B, N), dev)
    _check(workspace, "workspace", device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    with _on(dev):
        st = lib().spec_verify_tree_greedy(
            _ptr(target_logits), _ptr(tree_tokens), _ptr(tree_parents), _ptr(tree_size),
            _ptr(out_path), _ptr(out_path_len), _ptr(out_tokens), _ptr(out_pred), B, N, V,
            _dtype_code(target_logits), _ptr(workspace), ws_bytes, _stream_handle(stream, dev))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_tree_greedy")


def spec_verify_kv_rollback(prefix_len, draft_len, out_num_emitted, drafter_len_in, target_len_out,
                            drafter_len_out, cache=None, gamma_max=None, stream=None) -> None:
    """Calls the C ABI spec_verify_kv_rollback on torch tensors. cache: an optional [B, L, ...]
    contiguous tensor whose trailing dimensions form one entry; its dropped entries are zeroed."""
    import torch
    B = prefix_len.shape[0]
    dev = prefix_len.device
    for name, t in (("prefix_len", prefix_len), ("draft_len", draft_len),
                    ("out_num_emitted", out_num_emitted), ("drafter_len_in", drafter_len_in),
                    ("target_len_out", target_len_out), ("drafter_len_out", drafter_len_out)):
        _check(t, name, torch.int32, (B,), dev)
    if gamma_max is None:
        raise ValueError("gamma_max is required")
    stride = entry = entries = 0
    if cache is not None:
        _check(cache, "cache", device=dev)
        entries = cache.shape[1]
        entry = cache[0, 0].numel() * cache.element_size()
        stride = cache[0].numel() * cache.element_size()
    with _on(dev):
        st = lib().spec_verify_kv_rollback(
            _ptr(prefix_len), _ptr(draft_len), _ptr(out_num_emitted), _ptr(drafter_len_in),
            _ptr(target_len_out), _ptr(drafter_len_out), _ptr(cache), stride, entry, entries, B,
            gamma_max, _stream_handle(stream, dev))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_kv_rollback")


def verify_tree(target_logits, tree_tokens, tree_parents, tree_size=None, stream=None):
    """Allocates the outputs, runs spec_verify_tree_greedy and returns
    (out_path [B, N], out_path_len [B], out_tokens [B, N+1], out_pred [B, N])."""
    import torch
    B, N, V = target_logits.shape
    dev = target_logits.device
    out_path = torch.empty((B, N), dtype=torch.int32, device=dev)
    out_len = torch.empty((B,), dtype=torch.int32, device=dev)
    out_tokens = torch.empty((B, N + 1), dtype=torch.int32, device=dev)
    out_pred = torch.empty((B, N), dtype=torch.int32, device=dev)
    ws = workspace_for(B, N - 1, V, _dtype_code(target_logits), dev, stream)
    spec_verify_tree_greedy(target_logits, tree_tokens, tree_parents, tree_size, out_path, out_len,
                            out_tokens, out_pred, ws, stream)
    return out_path, out_len, out_tokens, out_pred


def spec_verify(target_logits, draft_logits, draft_tokens, draft_len, temperature, uniforms,
                out_tokens, out_num_emitted, out_alpha, workspace, stream=None) -> None:
    """Calls the C ABI spec_verify on torch tensors (see spec_verify_ex)."""
    spec_verify_ex(target_logits, draft_logits, draft_tokens, draft_len, temperature, uniforms,
                   out_tokens, out_num_emitted, out_alpha, None, None, workspace, stream)


_ws_cache = {}


def workspace_for(B, G, V, dtype_code, device, stream=None, filtered=False):
    """A zero-initialised workspace cached per (device, stream), grown on demand (``filtered``: the
    size with which spec_verify_filtered also verifies from kept lists). Calls leave it zeroed, so
    it is reused without clearing; it must not serve two calls in flight at once."""
    import torch
    need = (spec_verify_filtered_workspace_size if filtered else spec_verify_workspace_size)(
        B, G, V, dtype_code)
    key = (str(device), _stream_handle(stream, device))
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def verify(target_logits, draft_logits, draft_tokens, draft_len, temperature, uniforms,
           with_probs=False, stream=None, onehot=False, top_k=None, top_p=None):
    """Allocates the outputs, runs spec_verify(_ex) (or spec_verify_onehot when ``onehot``: the
    drafts are one-hot and draft_logits is ignored; or spec_verify_filtered when ``top_k`` or
    ``top_p`` is given) and returns
    (out_tokens [B, G+1], out_num_emitted [B], out_alpha [B, G][, out_p, out_q])."""
    import torch
    B, G1, V = target_logits.shape
    G = G1 - 1
    dev = target_logits.device
    out_tokens = torch.empty((B, G1), dtype=torch.int32, device=dev)
    out_num = torch.empty((B,), dtype=torch.int32, device=dev)
    out_alpha = torch.empty((B, G), dtype=torch.float32, device=dev)
    out_p = torch.empty((B, G), dtype=torch.float32, device=dev) if with_probs else None
    out_q = torch.empty((B, G), dtype=torch.float32, device=dev) if with_probs else None
    filtered = top_k is not None or top_p is not None
    ws = workspace_for(B, G, V, _dtype_code(target_logits), dev, stream, filtered=filtered)
    if filtered:
        if onehot:
            raise ValueError("filtering with one-hot drafts is not supported")
        spec_verify_filtered(target_logits, draft_logits, draft_tokens, draft_len, temperature,
                             top_k, top_p, uniforms, out_tokens, out_num, out_alpha, out_p, out_q,
                             ws, stream)
    elif onehot:
        spec_verify_onehot(target_logits, draft_tokens, draft_len, temperature, uniforms,
                           out_tokens, out_num, out_alpha, out_p, out_q, ws, stream)
    else:
        spec_verify_ex(target_logits, draft_logits, draft_tokens, draft_len, temperature, uniforms,
                       out_tokens, out_num, out_alpha, out_p, out_q, ws, stream)
    if with_probs:
        return out_tokens, out_num, out_alpha, out_p, out_q
    return out_tokens, out_num, out_alpha
