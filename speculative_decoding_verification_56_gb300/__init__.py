"""GB300-native batched draft-token verification for speculative decoding.

Thin ctypes binding over ``libspecverify.so`` (C ABI in ``include/spec_verify.h``).
Every step of verification runs in the library's CUDA kernels; this module only
marshals torch CUDA tensors (device memory, streams) into pointers and sizes.
There is no CPU fallback: without the compiled library every call raises.

Entry points (same names as the C ABI):

* :func:`spec_verify_sample`      -- rejection-sampling verification of chains
* :func:`spec_verify_greedy`      -- greedy verification of chains
* :func:`spec_verify_tree_greedy` -- greedy verification of draft trees
* :func:`spec_tree_attention_mask` -- ancestor bitmask + depth of draft trees
* :func:`spec_kv_commit_path`     -- move the accepted path's KV entries into place
* :func:`spec_lm_head_verify_greedy` -- LM head (tcgen05 GEMM) fused with greedy verification
* :func:`spec_lm_head_verify_sample` -- LM head (tcgen05 GEMM) fused with sampling verification
* :func:`spec_tree_grow`          -- EAGLE-2 dynamic draft-tree growth
* :func:`spec_verify_workspace_bytes`, :func:`spec_verify_read_flags`,
  :func:`spec_verify_launch_count`, :func:`spec_status_string`

Convenience wrappers that also allocate outputs and a workspace with torch:
:func:`verify_sample`, :func:`verify_greedy`, :func:`verify_tree_greedy`,
:func:`tree_attention_mask`.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

SPEC_OK = 0
SPEC_ERR_INVALID_ARG = 1
SPEC_ERR_ALIGNMENT = 2
SPEC_ERR_WORKSPACE = 3
SPEC_ERR_CUDA = 4
SPEC_ERR_TOO_LARGE = 5
SPEC_NOALLOC_SCRATCH_BYTES = 4 << 20
SPEC_DTYPE_F32 = 0
SPEC_DTYPE_BF16 = 1
SPEC_MODE_SAMPLE = 0
SPEC_MODE_GREEDY = 1
SPEC_MODE_TREE_GREEDY = 2
SPEC_MODE_TREE_MASK = 3
SPEC_MODE_KV_COMMIT = 4
SPEC_MODE_LM_HEAD_GREEDY = 5
SPEC_MODE_TREE_GROW = 6
SPEC_MODE_LM_HEAD_SAMPLE = 7
SPEC_LM_MAX_D = 8192
SPEC_FLAG_TOKEN_RANGE = 1
SPEC_FLAG_BAD_PARENT = 2
SPEC_FLAG_DEPTH = 4
SPEC_FLAG_RESIDUAL_FALLBACK = 8
SPEC_FLAG_TIMEOUT = 16
SPEC_FLAG_BAD_PATH = 32

_lock = threading.Lock()
_lib = None


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {spec_status_string(status)} (status {status})")


def load_library(path: str = LIB_PATH):
    """Load the compiled C-ABI library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with "
                "`python -m speculative_decoding_verification_56_gb300.build`")
        lib = ctypes.CDLL(path)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.spec_verify_workspace_bytes.argtypes = [I, I, I, I, I]
        lib.spec_verify_workspace_bytes.restype = Z
        lib.spec_verify_sample.argtypes = [P, P, I, P, P, P, F, I, I, I, P, P, P, P, P, P, Z, P]
        lib.spec_verify_sample.restype = I
        lib.spec_verify_greedy.argtypes = [P, I, P, I, I, I, P, P, P, Z, P]
        lib.spec_verify_greedy.restype = I
        lib.spec_verify_tree_greedy.argtypes = [P, I, P, P, I, I, I, I, P, P, P, P, Z, P]
        lib.spec_verify_tree_greedy.restype = I
        lib.spec_verify_greedy_noalloc.argtypes = [P, I, P, I, I, I, P, P, P]
        lib.spec_verify_greedy_noalloc.restype = I
        lib.spec_verify_selftest_exp2.argtypes = [P, P, P, I, P]
        lib.spec_verify_selftest_exp2.restype = I
        lib.spec_tree_attention_mask.argtypes = [P, I, I, P, P, P, Z, P]
        lib.spec_tree_attention_mask.restype = I
        LL = ctypes.c_longlong
        lib.spec_kv_commit_path.argtypes = [P, I, I, LL, LL, I, I, I, P, P, P, I, P, P, Z, P]
        lib.spec_kv_commit_path.restype = I
        lib.spec_lm_head_verify_greedy.argtypes = [P, P, P, I, I, I, I, P, P, P, Z, P]
        lib.spec_lm_head_verify_greedy.restype = I
        lib.spec_lm_head_verify_sample.argtypes = [P, P, P, P, P, P, F, I, I, I, I, P, P, P, P, P,
                                                   P, Z, P]
        lib.spec_lm_head_verify_sample.restype = I
        lib.spec_tree_grow.argtypes = [P, I, F, I, I, I, I, I, P, P, P, P, P, Z, P]
        lib.spec_tree_grow.restype = I
        lib.spec_verify_read_flags.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), I, P]
        lib.spec_verify_read_flags.restype = I
        lib.spec_verify_launch_count.argtypes = []
        lib.spec_verify_launch_count.restype = ctypes.c_uint64
        lib.spec_verify_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        lib.spec_verify_set_wait_limit_ns.restype = None
        lib.spec_status_string.argtypes = [I]
        lib.spec_status_string.restype = ctypes.c_char_p
        lib.spec_verify_abi_version.argtypes = []
        lib.spec_verify_abi_version.restype = I
        _lib = lib
        return lib


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return SPEC_DTYPE_BF16
    if t.dtype == torch.float32:
        return SPEC_DTYPE_F32
    raise TypeError(f"logits must be torch.bfloat16 or torch.float32, got {t.dtype}")


def _dev(t, name, dtype=None, optional=False):
    """Pointer of a contiguous CUDA tensor (None -> NULL when optional)."""
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream_ptr(stream):
    if stream is None:
        return _torch().cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status, where):
    if status != SPEC_OK:
        raise SpecVerifyError(status, where)


# ---------------------------------------------------------------------------
# C-ABI entry points
# ---------------------------------------------------------------------------

def spec_status_string(status: int) -> str:
    try:
        return load_library().spec_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def spec_verify_workspace_bytes(mode: int, B: int, k_or_N: int, V: int, dtype: int) -> int:
    return int(load_library().spec_verify_workspace_bytes(mode, B, k_or_N, V, dtype))


def spec_verify_launch_count() -> int:
    return int(load_library().spec_verify_launch_count())


def spec_verify_abi_version() -> int:
    return int(load_library().spec_verify_abi_version())


def spec_verify_set_wait_limit_ns(limit_ns: int) -> None:
    """Limit of the verification kernels' waits on their bulk copies for calls
    enqueued afterwards (0 restores the default 0.2 s); a diagnostic control
    for testing the timeout path."""
    load_library().spec_verify_set_wait_limit_ns(int(limit_ns))


def spec_verify_sample(target_logits, draft_logits, draft_tokens, u_accept, u_sample,
                       temperature, accepted_len, out_tokens, p_out, q_out, resid_mass,
                       workspace, stream=None):
    """Rejection-sampling verification (C ABI ``spec_verify_sample``).

    target_logits [B, k+1, V] and draft_logits [B, k, V] (bf16 or fp32);
    draft_tokens int32 [B, k]; u_accept float32 [B, k]; u_sample float32 [B].
    Outputs (preallocated CUDA tensors): accepted_len int32 [B], out_tokens
    int32 [B, k+1], p_out/q_out float32 [B, k], resid_mass float32 [B].
    workspace: uint8 CUDA tensor of at least spec_verify_workspace_bytes() bytes.
    """
    torch = _torch()
    B, k1, V = target_logits.shape
    k = k1 - 1
    dt = _dtype_code(target_logits)
    if k > 0 and (draft_logits is None or draft_logits.dtype != target_logits.dtype
                  or tuple(draft_logits.shape) != (B, k, V)):
        raise ValueError("draft_logits must be [B, k, V] with the target's dtype")
    st = load_library().spec_verify_sample(
        _dev(target_logits, "target_logits"),
        _dev(draft_logits, "draft_logits", optional=k == 0), dt,
        _dev(draft_tokens, "draft_tokens", torch.int32, optional=k == 0),
        _dev(u_accept, "u_accept", torch.float32, optional=k == 0),
        _dev(u_sample, "u_sample", torch.float32), float(temperature), B, k, V,
        _dev(accepted_len, "accepted_len", torch.int32),
        _dev(out_tokens, "out_tokens", torch.int32),
        _dev(p_out, "p_out", torch.float32, optional=k == 0),
        _dev(q_out, "q_out", torch.float32, optional=k == 0),
        _dev(resid_mass, "resid_mass", torch.float32),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream))
    _check(st, "spec_verify_sample")


def spec_verify_greedy(target_logits, draft_tokens, accepted_len, out_tokens, workspace,
                       stream=None):
    """Greedy verification (C ABI ``spec_verify_greedy``)."""
    torch = _torch()
    B, k1, V = target_logits.shape
    k = k1 - 1
    st = load_library().spec_verify_greedy(
        _dev(target_logits, "target_logits"), _dtype_code(target_logits),
        _dev(draft_tokens, "draft_tokens", torch.int32, optional=k == 0), B, k, V,
        _dev(accepted_len, "accepted_len", torch.int32),
        _dev(out_tokens, "out_tokens", torch.int32),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream))
    _check(st, "spec_verify_greedy")


def spec_verify_greedy_noalloc(target_logits, draft_tokens, accepted_len, out_tokens,
                               stream=None):
    """Greedy verification on the library's fixed device scratch (C ABI
    ``spec_verify_greedy_noalloc``): for callers that cannot allocate device
    memory when they verify.  Calls sharing the scratch must not overlap."""
    torch = _torch()
    B, k1, V = target_logits.shape
    k = k1 - 1
    st = load_library().spec_verify_greedy_noalloc(
        _dev(target_logits, "target_logits"), _dtype_code(target_logits),
        _dev(draft_tokens, "draft_tokens", torch.int32, optional=k == 0), B, k, V,
        _dev(accepted_len, "accepted_len", torch.int32),
        _dev(out_tokens, "out_tokens", torch.int32), _stream_ptr(stream))
    _check(st, "spec_verify_greedy_noalloc")


def spec_verify_tree_greedy(target_logits, node_tokens, parents, max_depth, accepted_len,
                            path_nodes, out_tokens, workspace, stream=None):
    """Draft-tree greedy verification (C ABI ``spec_verify_tree_greedy``)."""
    torch = _torch()
    B, N, V = target_logits.shape
    st = load_library().spec_verify_tree_greedy(
        _dev(target_logits, "target_logits"), _dtype_code(target_logits),
        _dev(node_tokens, "node_tokens", torch.int32), _dev(parents, "parents", torch.int32),
        B, N, V, int(max_depth),
        _dev(accepted_len, "accepted_len", torch.int32),
        _dev(path_nodes, "path_nodes", torch.int32),
        _dev(out_tokens, "out_tokens", torch.int32),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream))
    _check(st, "spec_verify_tree_greedy")


def spec_tree_attention_mask(parents, mask, depth, workspace, stream=None):
    """Tree attention mask (C ABI ``spec_tree_attention_mask``): ``mask``
    int32/uint32-sized [B, N, ceil(N/32)] words, ``depth`` int32 [B, N] or
    None."""
    torch = _torch()
    B, N = parents.shape
    st = load_library().spec_tree_attention_mask(
        _dev(parents, "parents", torch.int32), B, N, _dev(mask, "mask"),
        _dev(depth, "depth", torch.int32, optional=True),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream))
    _check(st, "spec_tree_attention_mask")


def spec_kv_commit_path(cache, base_len, accepted_len, path_nodes, N, new_len, workspace,
                        stream=None):
    """KV commit of the accepted path (C ABI ``spec_kv_commit_path``), in
    place.  ``cache``: contiguous CUDA tensor [planes, B, L, ...] (one entry =
    the trailing dimensions of one position)."""
    torch = _torch()
    planes, B, L = cache.shape[:3]
    entry = cache[0, 0, 0].numel() * cache.element_size()
    st = load_library().spec_kv_commit_path(
        _dev(cache, "cache"), B, planes, B * L * entry, L * entry, entry, L, int(N),
        _dev(base_len, "base_len", torch.int32), _dev(accepted_len, "accepted_len", torch.int32),
        _dev(path_nodes, "path_nodes", torch.int32), path_nodes.shape[1] - 1,
        _dev(new_len, "new_len", torch.int32),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream))
    _check(st, "spec_kv_commit_path")


def spec_lm_head_verify_greedy(hidden, w_lm, draft_tokens, accepted_len, out_tokens, workspace,
                               stream=None):
    """LM head fused with greedy verification (C ABI
    ``spec_lm_head_verify_greedy``): ``hidden`` bf16 [B*(k+1), d], ``w_lm``
    bf16 [V, d], ``draft_tokens`` int32 [B, k]."""
    torch = _torch()
    B, k = draft_tokens.shape
    rows, d = hidden.shape
    V = w_lm.shape[0]
    if rows != B * (k + 1) or w_lm.shape[1] != d:
        raise ValueError("hidden must be [B*(k+1), d] and w_lm [V, d]")
    st = load_library().spec_lm_head_verify_greedy(
        _dev(hidden, "hidden", torch.bfloat16), _dev(w_lm, "w_lm", torch.bfloat16),
        _dev(draft_tokens, "draft_tokens", torch.int32), B, k, d, V,
        _dev(accepted_len, "accepted_len", torch.int32),
        _dev(out_tokens, "out_tokens", torch.int32),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream))
    _check(st, "spec_lm_head_verify_greedy")


def spec_lm_head_verify_sample(h_target, h_draft, w_lm, draft_tokens, u_accept, u_sample,
                               temperature, accepted_len, out_tokens, p_out, q_out, resid_mass,
                               workspace, stream=None):
    """LM head fused with sampling verification (C ABI
    ``spec_lm_head_verify_sample``): ``h_target`` bf16 [B*(k+1), d],
    ``h_draft`` bf16 [B*k, d], ``w_lm`` bf16 [V, d], the rest as
    :func:`spec_verify_sample`."""
    torch = _torch()
    B, k = draft_tokens.shape
    rows, d = h_target.shape
    V = w_lm.shape[0]
    if rows != B * (k + 1) or w_lm.shape[1] != d:
        raise ValueError("h_target must be [B*(k+1), d] and w_lm [V, d]")
    if k > 0 and tuple(h_draft.shape) != (B * k, d):
        raise ValueError("h_draft must be [B*k, d]")
    st = load_library().spec_lm_head_verify_sample(
        _dev(h_target, "h_target", torch.bfloat16),
        _dev(h_draft, "h_draft", torch.bfloat16, optional=k == 0),
        _dev(w_lm, "w_lm", torch.bfloat16),
        _dev(draft_tokens, "draft_tokens", torch.int32, optional=k == 0),
        _dev(u_accept, "u_accept", torch.float32, optional=k == 0),
        _dev(u_sample, "u_sample", torch.float32), float(temperature), B, k, d, V,
        _dev(accepted_len, "accepted_len", torch.int32),
        _dev(out_tokens, "out_tokens", torch.int32),
        _dev(p_out, "p_out", torch.float32, optional=k == 0),
        _dev(q_out, "q_out", torch.float32, optional=k == 0),
        _dev(resid_mass, "resid_mass", torch.float32),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream))
    _check(st, "spec_lm_head_verify_sample")


def spec_tree_grow(draft_logits, temperature, M, tokens, parents, depth, values, workspace,
                   stream=None):
    """EAGLE-2 tree growth (C ABI ``spec_tree_grow``): ``draft_logits``
    [B, D, K, V] bf16 or fp32; outputs [B, M+1]."""
    torch = _torch()
    B, D, K, V = draft_logits.shape
    st = load_library().spec_tree_grow(
        _dev(draft_logits, "draft_logits"), _dtype_code(draft_logits), float(temperature),
        B, D, K, V, int(M), _dev(tokens, "tokens", torch.int32),
        _dev(parents, "parents", torch.int32), _dev(depth, "depth", torch.int32),
        _dev(values, "values", torch.float32),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream))
    _check(st, "spec_tree_grow")


def spec_verify_read_flags(workspace, clear: bool = True, stream=None) -> int:
    """Device flag bits recorded in ``workspace`` (synchronises the stream)."""
    out = ctypes.c_uint32(0)
    st = load_library().spec_verify_read_flags(_dev(workspace, "workspace"), ctypes.byref(out),
                                               1 if clear else 0, _stream_ptr(stream))
    _check(st, "spec_verify_read_flags")
    return int(out.value)


# ---------------------------------------------------------------------------
# convenience: allocate outputs + workspace with torch, then call the C ABI
# ---------------------------------------------------------------------------

def alloc_workspace(mode: int, B: int, k_or_N: int, V: int, dtype: int, device="cuda"):
    """Zero-filled workspace for one call shape (reusable for any smaller one)."""
    n = spec_verify_workspace_bytes(mode, B, k_or_N, V, dtype)
    if n == 0:
        raise ValueError("shape outside the library's limits")
    return _torch().zeros(n, dtype=_torch().uint8, device=device)


def verify_sample(target_logits, draft_logits, draft_tokens, u_accept, u_sample, temperature,
                  workspace=None, stream=None):
    torch = _torch()
    B, k1, V = target_logits.shape
    k = k1 - 1
    dev = target_logits.device
    if workspace is None:
        workspace = alloc_workspace(SPEC_MODE_SAMPLE, B, k, V, _dtype_code(target_logits), dev)
    out = dict(accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
               out_tokens=torch.empty(B, k + 1, dtype=torch.int32, device=dev),
               p=torch.empty(B, k, dtype=torch.float32, device=dev),
               q=torch.empty(B, k, dtype=torch.float32, device=dev),
               resid_mass=torch.empty(B, dtype=torch.float32, device=dev))
    spec_verify_sample(target_logits, draft_logits, draft_tokens, u_accept, u_sample,
                       temperature, out["accepted_len"], out["out_tokens"], out["p"], out["q"],
                       out["resid_mass"], workspace, stream)
    return out


def verify_greedy(target_logits, draft_tokens, workspace=None, stream=None):
    torch = _torch()
    B, k1, V = target_logits.shape
    dev = target_logits.device
    if workspace is None:
        workspace = alloc_workspace(SPEC_MODE_GREEDY, B, k1 - 1, V, _dtype_code(target_logits),
                                    dev)
    out = dict(accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
               out_tokens=torch.empty(B, k1, dtype=torch.int32, device=dev))
    spec_verify_greedy(target_logits, draft_tokens, out["accepted_len"], out["out_tokens"],
                       workspace, stream)
    return out


def verify_tree_greedy(target_logits, node_tokens, parents, max_depth, workspace=None,
                       stream=None):
    torch = _torch()
    B, N, V = target_logits.shape
    dev = target_logits.device
    if workspace is None:
        workspace = alloc_workspace(SPEC_MODE_TREE_GREEDY, B, N, V,
                                    _dtype_code(target_logits), dev)
    W = int(max_depth) + 1
    out = dict(accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
               path_nodes=torch.empty(B, W, dtype=torch.int32, device=dev),
               out_tokens=torch.empty(B, W, dtype=torch.int32, device=dev))
    spec_verify_tree_greedy(target_logits, node_tokens, parents, max_depth,
                            out["accepted_len"], out["path_nodes"], out["out_tokens"],
                            workspace, stream)
    return out


def tree_attention_mask(parents, workspace=None, stream=None):
    """Ancestor bitmask and depth of B draft trees: returns ``(mask, depth)``
    with mask int32 [B, N, ceil(N/32)] (the bit patterns of the C ABI's
    uint32 words) and depth int32 [B, N]."""
    torch = _torch()
    B, N = parents.shape
    dev = parents.device
    if workspace is None:
        workspace = alloc_workspace(SPEC_MODE_TREE_MASK, B, N, 1, SPEC_DTYPE_F32, dev)
    mask = torch.empty(B, N, (N + 31) // 32, dtype=torch.int32, device=dev)
    depth = torch.empty(B, N, dtype=torch.int32, device=dev)
    spec_tree_attention_mask(parents, mask, depth, workspace, stream)
    return mask, depth


def lm_head_verify_greedy(hidden, w_lm, draft_tokens, workspace=None, stream=None):
    """Greedy verification straight from hidden states and the LM head."""
    torch = _torch()
    B, k = draft_tokens.shape
    dev = hidden.device
    if workspace is None:
        workspace = alloc_workspace(SPEC_MODE_LM_HEAD_GREEDY, B, k, w_lm.shape[0],
                                    SPEC_DTYPE_BF16, dev)
    out = dict(accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
               out_tokens=torch.empty(B, k + 1, dtype=torch.int32, device=dev))
    spec_lm_head_verify_greedy(hidden, w_lm, draft_tokens, out["accepted_len"],
                               out["out_tokens"], workspace, stream)
    return out


def lm_head_verify_sample(h_target, h_draft, w_lm, draft_tokens, u_accept, u_sample, temperature,
                          workspace=None, stream=None):
    """Sampling verification straight from hidden states, drafted features
    and the LM head; returns the outputs of :func:`verify_sample`."""
    torch = _torch()
    B, k = draft_tokens.shape
    dev = h_target.device
    if workspace is None:
        workspace = alloc_workspace(SPEC_MODE_LM_HEAD_SAMPLE, B, k, w_lm.shape[0],
                                    SPEC_DTYPE_BF16, dev)
    i32 = dict(dtype=torch.int32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    out = dict(accepted_len=torch.empty(B, **i32), out_tokens=torch.empty(B, k + 1, **i32),
               p=torch.empty(B, k, **f32), q=torch.empty(B, k, **f32),
               resid_mass=torch.empty(B, **f32))
    spec_lm_head_verify_sample(h_target, h_draft, w_lm, draft_tokens, u_accept, u_sample,
                               temperature, out["accepted_len"], out["out_tokens"], out["p"],
                               out["q"], out["resid_mass"], workspace, stream)
    return out


def tree_grow(draft_logits, temperature, M, workspace=None, stream=None):
    """Grow B draft trees; returns dict(tokens, parents, depth, values) [B, M+1]."""
    torch = _torch()
    B, D, K, V = draft_logits.shape
    dev = draft_logits.device
    if workspace is None:
        workspace = alloc_workspace(SPEC_MODE_TREE_GROW, B, K, V, _dtype_code(draft_logits), dev)
    i32 = dict(dtype=torch.int32, device=dev)
    out = dict(tokens=torch.empty(B, M + 1, **i32), parents=torch.empty(B, M + 1, **i32),
               depth=torch.empty(B, M + 1, **i32),
               values=torch.empty(B, M + 1, dtype=torch.float32, device=dev))
    spec_tree_grow(draft_logits, temperature, M, out["tokens"], out["parents"], out["depth"],
                   out["values"], workspace, stream)
    return out


def to_device_logits(arr, dtype: str, device="cuda"):
    """numpy logits (float32, or uint16 bf16 bits) -> torch CUDA tensor."""
    import numpy as np
    torch = _torch()
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32))
    return t.to(device)
