"""Thin Python binding of libspecverify (ctypes).

Argument marshalling only: each function checks tensor placement, dtype and shape, takes
element strides and the current CUDA stream from PyTorch, allocates the outputs and the
workspace with PyTorch's caching allocator, and calls the C entry point of the same name.
Every step of the verification runs in the library's CUDA kernels; there is no CPU path.
If the shared library is missing the first call raises, telling how to build it.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

SV_OK = 0
(MODE_SAMPLE, MODE_GREEDY, MODE_TREE, MODE_ROW_STATS, MODE_TREE_SAMPLE, MODE_SAMPLE_LAZY, MODE_TYPICAL,
 MODE_SAMPLE_ONEHOT) = range(8)
FP32, BF16 = 0, 1

_lock = threading.Lock()
_lib = None


class SpecVerifyError(RuntimeError):
    pass


def library_path() -> str:
    """The product library, or the build named by SV_LIBRARY (e.g. the bounds-checked one)."""
    return os.environ.get("SV_LIBRARY") or _build.LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load libspecverify.so (built in-tree by __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise SpecVerifyError(
                f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        P, i64, i32, u64, f32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64,
                                     ctypes.c_float, ctypes.c_size_t)
        lib.spec_verify_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        lib.spec_verify_workspace_size.restype = sz
        lib.spec_verify_sample.argtypes = [P, i64, i64, P, i64, i64, i32, i32, i32, i32, P, f32, u64,
                                           u64, P, P, P, sz, P]
        lib.spec_verify_sample.restype = i32
        lib.spec_verify_greedy.argtypes = [P, i64, i64, i32, i32, i32, i32, P, P, P, P, sz, P]
        lib.spec_verify_greedy.restype = i32
        lib.spec_verify_tree_greedy.argtypes = [P, i64, i64, i32, i32, i32, i32, P, P, i32, P, P, P,
                                                P, sz, P]
        lib.spec_verify_tree_greedy.restype = i32
        lib.spec_verify_tree_sample.argtypes = [P, i64, i64, P, i64, i64, i32, i32, i32, i32, P, P, i32,
                                                f32, u64, u64, i32, P, P, P, P, sz, P]
        lib.spec_verify_tree_sample.restype = i32
        lib.spec_verify_sample_lazy.argtypes = [P, i64, i64, P, i64, i64, i32, i32, i32, i32, P, f32, u64,
                                                u64, P, P, P, sz, P]
        lib.spec_verify_sample_lazy.restype = i32
        lib.spec_verify_greedy_lazy.argtypes = [P, i64, i64, i32, i32, i32, i32, P, P, P, P]
        lib.spec_verify_greedy_lazy.restype = i32
        lib.spec_verify_typical.argtypes = [P, i64, i64, i32, i32, i32, i32, P, f32, f32, f32, u64, u64, P, P, P,
                                            sz, P]
        lib.spec_verify_typical.restype = i32
        lib.spec_verify_sample_onehot.argtypes = [P, i64, i64, i32, i32, i32, i32, P, f32, u64, u64, P, P, P, sz, P]
        lib.spec_verify_sample_onehot.restype = i32
        lib.spec_verify_tree_greedy_lazy.argtypes = [P, i64, i64, i32, i32, i32, i32, P, P, i32, P, P, P, P]
        lib.spec_verify_tree_greedy_lazy.restype = i32
        lib.spec_ngram_draft.argtypes = [P, i64, P, i32, i32, i32, i32, P, P, P]
        lib.spec_ngram_draft.restype = i32
        lib.spec_verify_row_stats.argtypes = [P, i64, i64, i32, i32, i32, i32, f32, P, P, P, sz, P]
        lib.spec_verify_row_stats.restype = i32
        lib.spec_verify_uniforms.argtypes = [u64, u64, i32, i32, i32, P, P]
        lib.spec_verify_uniforms.restype = i32
        lib.spec_verify_greedy_noalloc.argtypes = [P, i64, i64, i32, i32, i32, i32, P, P, P, P]
        lib.spec_verify_greedy_noalloc.restype = i32
        lib.spec_verify_status_offset.argtypes = [i32, i32, i32, i32, i32]
        lib.spec_verify_status_offset.restype = sz
        lib.spec_verify_wait_selftest.argtypes = [P, i32, ctypes.c_uint32, P]
        lib.spec_verify_wait_selftest.restype = i32
        lib.spec_verify_exp_df.argtypes = [P, P, i32, P, P, P]
        lib.spec_verify_exp_df.restype = i32
        lib.spec_verify_set_stage_events.argtypes = [P, i32]
        lib.spec_verify_set_stage_events.restype = i32
        lib.spec_verify_status_string.argtypes = [i32]
        lib.spec_verify_status_string.restype = ctypes.c_char_p
        lib.spec_verify_version.argtypes = []
        lib.spec_verify_version.restype = i32
        lib.spec_verify_check_word.argtypes = [P]
        lib.spec_verify_check_word.restype = i32
        lib.spec_verify_check_selftest.argtypes = [i64, i64]
        lib.spec_verify_check_selftest.restype = i32
        _lib = lib
        return lib


def _check(status: int, what: str):
    if status != SV_OK:
        msg = load_library().spec_verify_status_string(status).decode()
        raise SpecVerifyError(f"{what} failed with status {status}: {msg}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _logits3(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the verifier has no CPU path)")
    if t.dim() != 3 or (t.shape[2] > 1 and t.stride(2) != 1):
        raise ValueError(f"{name} must be [B, rows, V] with a contiguous last axis")
    return t.stride(0), t.stride(1)


def _ints(t: torch.Tensor, name: str, shape, dev=None) -> torch.Tensor:
    if not t.is_cuda or t.dtype != torch.int32:
        raise ValueError(f"{name} must be an int32 CUDA tensor")
    if dev is not None and t.device != dev:
        raise ValueError(f"{name} must be on {dev}, got {t.device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.contiguous()


def _out(t, name: str, shape, dev) -> torch.Tensor:
    """A caller-provided int32 output, checked (the kernels write it in place), or a new one."""
    if t is None:
        return torch.empty(tuple(shape), dtype=torch.int32, device=dev)
    if not t.is_cuda or t.device != dev or t.dtype != torch.int32 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous int32 tensor on {dev}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _like(t: torch.Tensor, ref: torch.Tensor, name: str):
    """A second logits tensor: on the target's device, with its dtype."""
    if t.device != ref.device or t.dtype != ref.dtype:
        raise ValueError(f"{name} must be on {ref.device} with dtype {ref.dtype}")


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def spec_verify_workspace_size(mode: int, B: int, rows: int, V: int, dtype: int) -> int:
    return int(load_library().spec_verify_workspace_size(mode, B, rows, V, dtype))


def _workspace(mode, B, rows, V, dtype, device, workspace):
    n = spec_verify_workspace_size(mode, B, rows, V, dtype)
    if workspace is None:
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=device)
    elif not workspace.is_cuda or workspace.device != device or not workspace.is_contiguous():
        raise ValueError(f"workspace must be a contiguous tensor on {device}")
    elif workspace.numel() * workspace.element_size() < n:
        raise ValueError(f"workspace too small: need {n} bytes")
    return workspace, workspace.numel() * workspace.element_size()


def spec_verify_sample(target: torch.Tensor, draft: torch.Tensor, draft_tokens: torch.Tensor,
                       temperature: float, seed: int, offset: int = 0, *, workspace=None,
                       accepted_len=None, out_tokens=None):
    """Sampling verification; returns (accepted_len [B] int32, out_tokens [B, gamma+1] int32)."""
    lib = load_library()
    tsb, tsr = _logits3(target, "target")
    B, G1, V = target.shape
    gamma = G1 - 1
    dt = _dtype_code(target)
    if gamma > 0:
        dsb, dsr = _logits3(draft, "draft")
        _like(draft, target, "draft")
        if tuple(draft.shape) != (B, gamma, V):
            raise ValueError("draft must be [B, gamma, V] with the target's dtype")
        dptr = draft.data_ptr()
        x = _ints(draft_tokens, "draft_tokens", (B, gamma), target.device)
        xptr = x.data_ptr()
    else:
        dsb = dsr = 0
        dptr = xptr = None
    dev = target.device
    accepted_len = _out(accepted_len, "accepted_len", (B,), dev)
    out_tokens = _out(out_tokens, "out_tokens", (B, G1), dev)
    ws, wsb = _workspace(MODE_SAMPLE, B, gamma, V, dt, dev, workspace)
    st = lib.spec_verify_sample(target.data_ptr(), tsb, tsr, dptr, dsb, dsr, dt, B, gamma, V, xptr,
                                float(temperature), int(seed) & (2**64 - 1),
                                int(offset) & (2**64 - 1), accepted_len.data_ptr(),
                                out_tokens.data_ptr(), ws.data_ptr(), wsb, _stream(dev))
    _check(st, "spec_verify_sample")
    return accepted_len, out_tokens


def spec_verify_greedy(target: torch.Tensor, draft_tokens: torch.Tensor, *, workspace=None,
                       accepted_len=None, out_tokens=None):
    """Greedy verification; returns (accepted_len [B], out_tokens [B, gamma+1])."""
    lib = load_library()
    tsb, tsr = _logits3(target, "target")
    B, G1, V = target.shape
    gamma = G1 - 1
    dt = _dtype_code(target)
    x = _ints(draft_tokens, "draft_tokens", (B, gamma), target.device) if gamma > 0 else None
    dev = target.device
    accepted_len = _out(accepted_len, "accepted_len", (B,), dev)
    out_tokens = _out(out_tokens, "out_tokens", (B, G1), dev)
    ws, wsb = _workspace(MODE_GREEDY, B, gamma, V, dt, dev, workspace)
    st = lib.spec_verify_greedy(target.data_ptr(), tsb, tsr, dt, B, gamma, V,
                                x.data_ptr() if x is not None else None, accepted_len.data_ptr(),
                                out_tokens.data_ptr(), ws.data_ptr(), wsb, _stream(dev))
    _check(st, "spec_verify_greedy")
    return accepted_len, out_tokens


def spec_verify_tree_greedy(target: torch.Tensor, parent: torch.Tensor, node_tokens: torch.Tensor,
                            max_depth: int, *, with_path: bool = True, workspace=None,
                            accepted_len=None, out_tokens=None, out_path=None):
    """Greedy token-tree verification; returns (accepted_len [B], out_tokens [B, D+1],
    out_path [B, D+1] or None)."""
    lib = load_library()
    tsb, tsr = _logits3(target, "target")
    B, N, V = target.shape
    dt = _dtype_code(target)
    par = _ints(parent, "parent", (N,), target.device)
    tok = _ints(node_tokens, "node_tokens", (B, N), target.device)
    dev = target.device
    W = int(max_depth) + 1
    accepted_len = _out(accepted_len, "accepted_len", (B,), dev)
    out_tokens = _out(out_tokens, "out_tokens", (B, W), dev)
    if with_path or out_path is not None:
        out_path = _out(out_path, "out_path", (B, W), dev)
    ws, wsb = _workspace(MODE_TREE, B, N, V, dt, dev, workspace)
    st = lib.spec_verify_tree_greedy(target.data_ptr(), tsb, tsr, dt, B, N, V, par.data_ptr(),
                                     tok.data_ptr(), int(max_depth), accepted_len.data_ptr(),
                                     out_tokens.data_ptr(),
                                     out_path.data_ptr() if out_path is not None else None,
                                     ws.data_ptr(), wsb, _stream(dev))
    _check(st, "spec_verify_tree_greedy")
    return accepted_len, out_tokens, out_path


def spec_verify_tree_sample(target: torch.Tensor, draft: torch.Tensor, parent: torch.Tensor,
                            node_tokens: torch.Tensor, max_depth: int, temperature: float, seed: int,
                            offset: int = 0, *, without_replacement: bool = False,
                            with_path: bool = True, workspace=None, accepted_len=None,
                            out_tokens=None, out_path=None):
    """Token-tree sampling verification (multi-round rejection); returns (accepted_len [B],
    out_tokens [B, D+1], out_path [B, D+1] or None)."""
    lib = load_library()
    tsb, tsr = _logits3(target, "target")
    dsb, dsr = _logits3(draft, "draft")
    B, N, V = target.shape
    dt = _dtype_code(target)
    _like(draft, target, "draft")
    if tuple(draft.shape) != (B, N, V):
        raise ValueError("draft must be [B, N, V] with the target's dtype")
    par = _ints(parent, "parent", (N,), target.device)
    tok = _ints(node_tokens, "node_tokens", (B, N), target.device)
    dev = target.device
    W = int(max_depth) + 1
    accepted_len = _out(accepted_len, "accepted_len", (B,), dev)
    out_tokens = _out(out_tokens, "out_tokens", (B, W), dev)
    if with_path or out_path is not None:
        out_path = _out(out_path, "out_path", (B, W), dev)
    ws, wsb = _workspace(MODE_TREE_SAMPLE, B, N, V, dt, dev, workspace)
    st = lib.spec_verify_tree_sample(target.data_ptr(), tsb, tsr, draft.data_ptr(), dsb, dsr, dt, B,
                                     N, V, par.data_ptr(), tok.data_ptr(), int(max_depth),
                                     float(temperature), int(seed) & (2**64 - 1),
                                     int(offset) & (2**64 - 1), int(bool(without_replacement)),
                                     accepted_len.data_ptr(), out_tokens.data_ptr(),
                                     out_path.data_ptr() if out_path is not None else None,
                                     ws.data_ptr(), wsb, _stream(dev))
    _check(st, "spec_verify_tree_sample")
    return accepted_len, out_tokens, out_path


def spec_verify_sample_lazy(target: torch.Tensor, draft: torch.Tensor, draft_tokens: torch.Tensor,
                            temperature: float, seed: int, offset: int = 0, *, workspace=None,
                            accepted_len=None, out_tokens=None):
    """Lazy sampling verification (reads rows up to the stop point); returns (accepted_len
    [B], out_tokens [B, gamma+1]) -- spec_verify_sample's outputs."""
    lib = load_library()
    tsb, tsr = _logits3(target, "target")
    B, G1, V = target.shape
    gamma = G1 - 1
    dt = _dtype_code(target)
    if gamma > 0:
        dsb, dsr = _logits3(draft, "draft")
        _like(draft, target, "draft")
        if tuple(draft.shape) != (B, gamma, V):
            raise ValueError("draft must be [B, gamma, V] with the target's dtype")
        dptr = draft.data_ptr()
        x = _ints(draft_tokens, "draft_tokens", (B, gamma), target.device)
        xptr = x.data_ptr()
    else:
        dsb = dsr = 0
        dptr = xptr = None
    dev = target.device
    accepted_len = _out(accepted_len, "accepted_len", (B,), dev)
    out_tokens = _out(out_tokens, "out_tokens", (B, G1), dev)
    ws, wsb = _workspace(MODE_SAMPLE_LAZY, B, gamma, V, dt, dev, workspace)
    st = lib.spec_verify_sample_lazy(target.data_ptr(), tsb, tsr, dptr, dsb, dsr, dt, B, gamma, V, xptr,
                                     float(temperature), int(seed) & (2**64 - 1),
                                     int(offset) & (2**64 - 1), accepted_len.data_ptr(),
                                     out_tokens.data_ptr(), ws.data_ptr(), wsb, _stream(dev))
    _check(st, "spec_verify_sample_lazy")
    return accepted_len, out_tokens


def spec_verify_typical(target: torch.Tensor, draft_tokens: torch.Tensor, temperature: float, epsilon: float,
                        delta: float, seed: int, offset: int = 0, *, workspace=None, accepted_len=None,
                        out_tokens=None):
    """Typical acceptance (threshold min(epsilon, delta exp(-H)) on the target probability);
    returns (accepted_len [B], out_tokens [B, gamma+1]) -- spec_verify_sample's outputs."""
    lib = load_library()
    tsb, tsr = _logits3(target, "target")
    B, G1, V = target.shape
    gamma = G1 - 1
    dt = _dtype_code(target)
    xptr = None
    if gamma > 0:
        x = _ints(draft_tokens, "draft_tokens", (B, gamma), target.device)
        xptr = x.data_ptr()
    dev = target.device
    accepted_len = _out(accepted_len, "accepted_len", (B,), dev)
    out_tokens = _out(out_tokens, "out_tokens", (B, G1), dev)
    ws, wsb = _workspace(MODE_TYPICAL, B, gamma, V, dt, dev, workspace)
    st = lib.spec_verify_typical(target.data_ptr(), tsb, tsr, dt, B, gamma, V, xptr, float(temperature),
                                 float(epsilon), float(delta), int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                                 accepted_len.data_ptr(), out_tokens.data_ptr(), ws.data_ptr(), wsb, _stream(dev))
    _check(st, "spec_verify_typical")
    return accepted_len, out_tokens


def spec_verify_sample_onehot(target: torch.Tensor, draft_tokens: torch.Tensor, temperature: float, seed: int,
                              offset: int = 0, *, workspace=None, accepted_len=None, out_tokens=None):
    """Sampling verification of drafts whose draft distribution is one-hot (a prompt-lookup
    drafter's); returns (accepted_len [B], out_tokens [B, gamma+1]) -- spec_verify_sample's
    outputs for draft rows that are -inf except at each draft."""
    lib = load_library()
    tsb, tsr = _logits3(target, "target")
    B, G1, V = target.shape
    gamma = G1 - 1
    dt = _dtype_code(target)
    xptr = None
    if gamma > 0:
        x = _ints(draft_tokens, "draft_tokens", (B, gamma), target.device)
        xptr = x.data_ptr()
    dev = target.device
    accepted_len = _out(accepted_len, "accepted_len", (B,), dev)
    out_tokens = _out(out_tokens, "out_tokens", (B, G1), dev)
    ws, wsb = _workspace(MODE_SAMPLE_ONEHOT, B, gamma, V, dt, dev, workspace)
    st = lib.spec_verify_sample_onehot(target.data_ptr(), tsb, tsr, dt, B, gamma, V, xptr, float(temperature),
                                       int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), accepted_len.data_ptr(),
                                       out_tokens.data_ptr(), ws.data_ptr(), wsb, _stream(dev))
    _check(st, "spec_verify_sample_onehot")
    return accepted_len, out_tokens


def spec_verify_greedy_lazy(target: torch.Tensor, draft_tokens: torch.Tensor, *, accepted_len=None,
                            out_tokens=None):
    """Lazy greedy verification (reads rows up to the first mismatch); returns
    spec_verify_greedy's outputs."""
    lib = load_library()
    tsb, tsr = _logits3(target, "target")
    B, G1, V = target.shape
    gamma = G1 - 1
    dt = _dtype_code(target)
    x = _ints(draft_tokens, "draft_tokens", (B, gamma), target.device) if gamma > 0 else None
    dev = target.device
    accepted_len = _out(accepted_len, "accepted_len", (B,), dev)
    out_tokens = _out(out_tokens, "out_tokens", (B, G1), dev)
    st = lib.spec_verify_greedy_lazy(target.data_ptr(), tsb, tsr, dt, B, gamma, V,
                                     x.data_ptr() if x is not None else None, accepted_len.data_ptr(),
                                     out_tokens.data_ptr(), _stream(dev))
    _check(st, "spec_verify_greedy_lazy")
    return accepted_len, out_tokens


def spec_verify_tree_greedy_lazy(target: torch.Tensor, parent: torch.Tensor, node_tokens: torch.Tensor,
                                 max_depth: int, *, with_path: bool = True, accepted_len=None,
                                 out_tokens=None, out_path=None):
    """Lazy greedy tree verification (reads the rows of accepted nodes only); returns
    spec_verify_tree_greedy's outputs."""
    lib = load_library()
    tsb, tsr = _logits3(target, "target")
    B, N, V = target.shape
    dt = _dtype_code(target)
    par = _ints(parent, "parent", (N,), target.device)
    tok = _ints(node_tokens, "node_tokens", (B, N), target.device)
    dev = target.device
    W = int(max_depth) + 1
    accepted_len = _out(accepted_len, "accepted_len", (B,), dev)
    out_tokens = _out(out_tokens, "out_tokens", (B, W), dev)
    if with_path or out_path is not None:
        out_path = _out(out_path, "out_path", (B, W), dev)
    st = lib.spec_verify_tree_greedy_lazy(target.data_ptr(), tsb, tsr, dt, B, N, V, par.data_ptr(),
                                          tok.data_ptr(), int(max_depth), accepted_len.data_ptr(),
                                          out_tokens.data_ptr(),
                                          out_path.data_ptr() if out_path is not None else None,
                                          _stream(dev))
    _check(st, "spec_verify_tree_greedy_lazy")
    return accepted_len, out_tokens, out_path


def spec_ngram_draft(history: torch.Tensor, lengths: torch.Tensor, n: int, k: int, pad: bool = False,
                     *, drafts=None, count=None):
    """Prompt-lookup drafts of a [B, T] int32 history with lengths [B]; returns (drafts
    [B, k] int32, -1 in unused slots, count [B] int32)."""
    lib = load_library()
    if not history.is_cuda or history.dim() != 2 or history.dtype != torch.int32 or history.stride(1) != 1:
        raise ValueError("history must be a [B, T] int32 CUDA tensor with contiguous rows")
    B, T = history.shape
    dev = history.device
    L = _ints(lengths, "lengths", (B,), dev)
    drafts = _out(drafts, "drafts", (B, max(int(k), 0)), dev)
    count = _out(count, "count", (B,), dev)
    st = lib.spec_ngram_draft(history.data_ptr(), history.stride(0), L.data_ptr(), B, int(n), int(k),
                              int(bool(pad)), drafts.data_ptr(), count.data_ptr(), _stream(dev))
    _check(st, "spec_ngram_draft")
    return drafts, count


def spec_verify_row_stats(logits: torch.Tensor, temperature: float = 1.0, *, workspace=None):
    """Test hook: (m, lse) per row of [B, rows, V] logits, fp32 [B, rows] each."""
    lib = load_library()
    sb, sr = _logits3(logits, "logits")
    B, R, V = logits.shape
    dt = _dtype_code(logits)
    dev = logits.device
    m = torch.empty((B, R), dtype=torch.float32, device=dev)
    lse = torch.empty((B, R), dtype=torch.float32, device=dev)
    ws, wsb = _workspace(MODE_ROW_STATS, B, R, V, dt, dev, workspace)
    st = lib.spec_verify_row_stats(logits.data_ptr(), sb, sr, dt, B, R, V, float(temperature),
                                   m.data_ptr(), lse.data_ptr(), ws.data_ptr(), wsb, _stream(dev))
    _check(st, "spec_verify_row_stats")
    return m, lse


def spec_verify_uniforms(seed: int, offset: int, B: int, positions: int, purpose: int,
                         device="cuda") -> torch.Tensor:
    """Test hook: the sampler's uniforms u(b, i, purpose) as a [B, positions] fp32 tensor."""
    lib = load_library()
    out = torch.empty((B, positions), dtype=torch.float32, device=device)
    st = lib.spec_verify_uniforms(int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), B, positions,
                                  purpose, out.data_ptr(), _stream(out.device))
    _check(st, "spec_verify_uniforms")
    return out


def call_status(workspace: torch.Tensor, mode: int, B: int, rows: int, V: int, dtype: int):
    """The device-side outcome of the last sampling call (mode MODE_SAMPLE, MODE_TREE_SAMPLE,
    MODE_SAMPLE_LAZY, MODE_TYPICAL or MODE_SAMPLE_ONEHOT; rows as for the workspace size)
    that used `workspace`: (sequences marked for the extended-precision pass, sequences
    redone, status, per-sequence marks as a numpy array).  Synchronises the device."""
    lib = load_library()
    off = lib.spec_verify_status_offset(mode, B, rows, V, dtype)
    if off == ctypes.c_size_t(-1).value:
        raise ValueError("bad mode or sizes")
    torch.cuda.synchronize(workspace.device)
    words = workspace.view(torch.uint8)[off:off + 4 * (8 + B)].clone().view(torch.int32).cpu().numpy()
    return int(words[0]), int(words[4]), int(words[3]), words[8:8 + B].copy()


def check_word():
    """The bounds-checked build's violation record (see spec_verify_check_word): (status,
    [site, index, extent, count]); status SV_ERR_UNSUPPORTED from the product build.  The
    site's high 16 bits are file_tag() of the source file's base name, the low 16 its line."""
    lib = load_library()
    info = (ctypes.c_int32 * 4)()
    st = lib.spec_verify_check_word(info)
    return int(st), [int(v) for v in info]


def check_selftest(index: int, extent: int) -> int:
    """Bounds-checked build: one check of index against extent on the device (no memory
    access); returns the launch status (SV_ERR_UNSUPPORTED from the product build)."""
    return int(load_library().spec_verify_check_selftest(index, extent))


def file_tag(name: str) -> int:
    """The 16-bit tag the bounds-checked build gives a source file (FNV-1a, folded)."""
    h = 2166136261
    for ch in name.encode():
        h = ((h ^ ch) * 16777619) & 0xFFFFFFFF
    return (h >> 16) ^ (h & 0xFFFF)


def wait_selftest(expected_arrivals: int, limit_us: int, device="cuda:0") -> int:
    """Test hook: one CTA waits for a flag (set by itself when expected_arrivals is 1) and
    meets the bounded grid barrier expecting `expected_arrivals` CTAs; returns the status
    word it leaves (4 = SV_ERR_TIMEOUT)."""
    lib = load_library()
    ctl = torch.zeros(8, dtype=torch.int32, device=device)
    _check(lib.spec_verify_wait_selftest(ctl.data_ptr(), int(expected_arrivals), int(limit_us),
                                         _stream(torch.device(device))), "spec_verify_wait_selftest")
    torch.cuda.synchronize(device)
    return int(ctl[3].item())


def spec_verify_exp_df(y_hi: torch.Tensor, y_lo: torch.Tensor):
    """Test hook: exp(y_hi + y_lo) in the re-draw's double-float arithmetic -> (hi, lo)."""
    lib = load_library()
    if y_hi.dtype != torch.float32 or y_lo.dtype != torch.float32 or y_hi.shape != y_lo.shape:
        raise ValueError("y_hi, y_lo: fp32 tensors of one shape")
    y_hi, y_lo = y_hi.contiguous(), y_lo.contiguous()
    out_hi, out_lo = torch.empty_like(y_hi), torch.empty_like(y_lo)
    _check(lib.spec_verify_exp_df(y_hi.data_ptr(), y_lo.data_ptr(), y_hi.numel(), out_hi.data_ptr(),
                                  out_lo.data_ptr(), _stream(y_hi.device)), "spec_verify_exp_df")
    return out_hi, out_lo


def set_stage_events(events) -> None:
    """Record the given torch.cuda.Event objects around the kernels of later calls made by
    this thread (see spec_verify_set_stage_events); None turns it off."""
    lib = load_library()
    if not events:
        _check(lib.spec_verify_set_stage_events(None, 0), "spec_verify_set_stage_events")
        return
    for e in events:
        if e.cuda_event == 0:
            e.record()  # torch creates the underlying event lazily
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(lib.spec_verify_set_stage_events(arr, len(events)), "spec_verify_set_stage_events")


def spec_verify_greedy_noalloc(target: torch.Tensor, draft_tokens: torch.Tensor, *,
                               accepted_len=None, out_tokens=None):
    """Greedy verification without a workspace: for callers that cannot allocate device
    memory while they run (the library's fixed device scratch holds the partials).  The
    outputs are allocated here unless passed in; the C call itself allocates nothing.
    Calls that overlap on the GPU share that scratch and must not run concurrently."""
    lib = load_library()
    tsb, tsr = _logits3(target, "target")
    B, G1, V = target.shape
    gamma = G1 - 1
    dt = _dtype_code(target)
    x = _ints(draft_tokens, "draft_tokens", (B, gamma), target.device) if gamma > 0 else None
    dev = target.device
    accepted_len = _out(accepted_len, "accepted_len", (B,), dev)
    out_tokens = _out(out_tokens, "out_tokens", (B, G1), dev)
    st = lib.spec_verify_greedy_noalloc(target.data_ptr(), tsb, tsr, dt, B, gamma, V,
                                        x.data_ptr() if x is not None else None,
                                        accepted_len.data_ptr(), out_tokens.data_ptr(),
                                        _stream(dev))
    _check(st, "spec_verify_greedy_noalloc")
    return accepted_len, out_tokens
