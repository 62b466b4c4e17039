"""The oracle for the speculative-decoding verification step.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference leg of ``bench.py`` may import this package.  The CUDA library
never calls it and shares no code with it.

This module is argument marshalling only: every step of the method lives in
``spec_oracle.c`` (plain fp64 C, compiled on demand with gcc), which cites the page
sections it follows.  Inputs are numpy arrays (or CPU torch tensors converted by the
caller); bf16 logits are passed as their raw 16-bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_FP32 = 0
DTYPE_BF16 = 1

FLAG_ACCEPT_NEAR_THRESHOLD = 1
FLAG_CDF_NEAR_BOUNDARY = 2
FLAG_RESIDUAL_NEAR_ZERO = 4
FLAG_RESIDUAL_FALLBACK = 8
FLAG_TREE_FIRST_MATCH_DIFFERS = 1


def compile_oracle(out_path: str = _LIB_PATH, src: str = _SRC) -> str:
    """Compile the oracle's C source into a shared object with plain gcc (C99, -O2)."""
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", out_path, src, "-lm"]
    subprocess.check_call(cmd)
    return out_path


def _bind(lib):
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    i32 = ctypes.c_int
    u64 = ctypes.c_uint64
    u32 = ctypes.c_uint32
    dbl = ctypes.c_double
    lib.oracle_philox4x32_10.argtypes = [P, P, P]
    lib.oracle_philox4x32_10.restype = None
    lib.oracle_uniform.argtypes = [u64, u64, u32, u32, u32]
    lib.oracle_uniform.restype = dbl
    lib.oracle_row_stats.argtypes = [P, i64, i64, i32, i32, i32, i32, dbl, P, P, P]
    lib.oracle_row_stats.restype = i32
    lib.oracle_verify_sample.argtypes = [P, i64, i64, P, i64, i64, i32, i32, i32, i32, i32,
                                         P, dbl, u64, u64, P, P, P, P]
    lib.oracle_verify_sample.restype = i32
    lib.oracle_exact_probs.argtypes = [P, P, i32, i32, P, dbl, P]
    lib.oracle_exact_probs.restype = i32
    lib.oracle_verify_greedy.argtypes = [P, i64, i64, i32, i32, i32, i32, P, P, P]
    lib.oracle_verify_greedy.restype = i32
    lib.oracle_verify_tree_greedy.argtypes = [P, i64, i64, i32, i32, i32, i32, P, P, i32,
                                              P, P, P, P]
    lib.oracle_verify_tree_greedy.restype = i32
    lib.oracle_verify_tree_sample.argtypes = [P, i64, i64, P, i64, i64, i32, i32, i32, i32, i32,
                                              P, P, i32, dbl, i32, u64, u64, P, P, P, P]
    lib.oracle_verify_tree_sample.restype = i32
    lib.oracle_exact_probs_tree.argtypes = [P, P, P, P, i32, i32, dbl, i32, P]
    lib.oracle_exact_probs_tree.restype = i32
    lib.oracle_ngram_draft.argtypes = [P, i64, P, i32, i32, i32, i32, P, P]
    lib.oracle_verify_typical.argtypes = [P, i64, i64, i32, i32, i32, i32, i32, P, dbl, dbl, dbl,
                                          u64, u64, P, P, P, P]
    lib.oracle_verify_typical.restype = ctypes.c_int
    lib.oracle_ngram_draft.restype = i32
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            compile_oracle()
        _lib = Oracle(_bind(ctypes.CDLL(_LIB_PATH)))
        return _lib


def variant(source_text: str, workdir: str) -> "Oracle":
    """Compile a modified copy of the oracle's source (a planted mistake, in tests that
    check that the pins catch it) and return it with the same interface."""
    src = os.path.join(workdir, "oracle_variant.c")
    with open(src, "w") as f:
        f.write(source_text)
    so = os.path.join(workdir, "liboracle_variant.so")
    compile_oracle(so, src)
    return Oracle(_bind(ctypes.CDLL(so)))


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _logits(arr):
    """Return (array, dtype code, element strides) for a numpy logits array.

    float32 arrays are read as fp32; uint16 arrays are read as raw bf16 bit patterns.
    The last axis must be contiguous; strides are returned in elements.
    """
    a = np.asarray(arr)
    if a.dtype == np.float32:
        code = DTYPE_FP32
    elif a.dtype == np.uint16:
        code = DTYPE_BF16
    else:
        raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {a.dtype}")
    if a.ndim != 3 or a.strides[2] != a.itemsize:
        raise ValueError("logits must be [B, rows, V] with a contiguous last axis")
    sb, sr = a.strides[0] // a.itemsize, a.strides[1] // a.itemsize
    return a, code, sb, sr


class Oracle:
    """The oracle's entry points over one loaded copy of the C code."""

    def __init__(self, lib):
        self.lib = lib

    def philox4x32_10(self, ctr, key) -> np.ndarray:
        c = np.asarray(ctr, dtype=np.uint32).copy()
        k = np.asarray(key, dtype=np.uint32).copy()
        out = np.zeros(4, dtype=np.uint32)
        self.lib.oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
        return out

    def uniform(self, seed: int, offset: int, b: int, i: int, purpose: int) -> float:
        return self.lib.oracle_uniform(seed, offset, b, i, purpose)

    def row_stats(self, logits, temperature: float = 1.0):
        """(m, lse, valid) for every row of [B, rows, V] logits, fp64."""
        a, code, sb, sr = _logits(logits)
        B, R, V = a.shape
        m = np.zeros(B * R, np.float64)
        lse = np.zeros(B * R, np.float64)
        valid = np.zeros(B * R, np.int32)
        rc = self.lib.oracle_row_stats(_ptr(a), sb, sr, code, B, R, V, float(temperature),
                                       _ptr(m), _ptr(lse), _ptr(valid))
        assert rc == 0
        return m.reshape(B, R), lse.reshape(B, R), valid.reshape(B, R).astype(bool)

    def verify_sample(self, target, draft, draft_tokens, temperature, seed, offset=0, b0=0,
                      diagnostics=False):
        """Sampling verification; returns (accepted_len[B], out_tokens[B, gamma+1], flags[B])
        and, with diagnostics=True, a [B, 4] array per sequence: final-draw kind (0 bonus,
        1 residual, 2 residual fell back to p, -1 invalid), its mass R, the distance of u'R
        to the nearer CDF boundary over R, and the smallest |u - p/q| of the accept tests."""
        t, code, tsb, tsr = _logits(target)
        B, G1, V = t.shape
        gamma = G1 - 1
        x = np.ascontiguousarray(np.asarray(draft_tokens, dtype=np.int32).reshape(B, gamma))
        if gamma > 0:
            d, dcode, dsb, dsr = _logits(draft)
            if dcode != code or d.shape != (B, gamma, V):
                raise ValueError("draft logits must match the target's dtype and be [B, gamma, V]")
            dptr = _ptr(d)
        else:
            dptr, dsb, dsr = None, 0, 0
        acc = np.zeros(B, np.int32)
        out = np.zeros((B, G1), np.int32)
        flags = np.zeros(B, np.int32)
        diag = np.zeros((B, 4), np.float64) if diagnostics else None
        rc = self.lib.oracle_verify_sample(_ptr(t), tsb, tsr, dptr, dsb, dsr, code, B, int(b0),
                                           gamma, V, _ptr(x), float(temperature), int(seed),
                                           int(offset), _ptr(acc), _ptr(out), _ptr(flags),
                                           _ptr(diag) if diagnostics else None)
        assert rc == 0
        return (acc, out, flags, diag) if diagnostics else (acc, out, flags)

    def exact_probs(self, t_logits, d_logits, draft_tokens, temperature) -> np.ndarray:
        """Enumeration mode: P(accepted_len = k, final token = j) as a [gamma+1, V] array."""
        t = np.ascontiguousarray(np.asarray(t_logits, dtype=np.float64))
        G1, V = t.shape
        gamma = G1 - 1
        d = np.ascontiguousarray(np.asarray(d_logits, dtype=np.float64).reshape(max(gamma, 0), V))
        x = np.ascontiguousarray(np.asarray(draft_tokens, dtype=np.int32).reshape(gamma))
        prob = np.zeros((G1, V), np.float64)
        rc = self.lib.oracle_exact_probs(_ptr(t), _ptr(d) if gamma else None, gamma, V, _ptr(x),
                                         float(temperature), _ptr(prob))
        if rc != 0:
            raise ValueError("invalid row or draft token")
        return prob

    def verify_greedy(self, target, draft_tokens):
        """Greedy verification; returns (accepted_len[B], out_tokens[B, gamma+1])."""
        t, code, tsb, tsr = _logits(target)
        B, G1, V = t.shape
        gamma = G1 - 1
        x = np.ascontiguousarray(np.asarray(draft_tokens, dtype=np.int32).reshape(B, gamma))
        acc = np.zeros(B, np.int32)
        out = np.zeros((B, G1), np.int32)
        rc = self.lib.oracle_verify_greedy(_ptr(t), tsb, tsr, code, B, gamma, V, _ptr(x),
                                           _ptr(acc), _ptr(out))
        assert rc == 0
        return acc, out

    def verify_tree_greedy(self, target, parent, node_tokens, max_depth):
        """Greedy tree verification; returns (accepted_len, out_tokens, out_path, flags)."""
        t, code, tsb, tsr = _logits(target)
        B, N, V = t.shape
        par = np.ascontiguousarray(np.asarray(parent, dtype=np.int32).reshape(N))
        toks = np.ascontiguousarray(np.asarray(node_tokens, dtype=np.int32).reshape(B, N))
        W = max_depth + 1
        acc = np.zeros(B, np.int32)
        out = np.zeros((B, W), np.int32)
        path = np.zeros((B, W), np.int32)
        flags = np.zeros(B, np.int32)
        rc = self.lib.oracle_verify_tree_greedy(_ptr(t), tsb, tsr, code, B, N, V, _ptr(par),
                                                _ptr(toks), int(max_depth), _ptr(acc), _ptr(out),
                                                _ptr(path), _ptr(flags))
        assert rc == 0
        return acc, out, path, flags


    def verify_tree_sample(self, target, draft, parent, node_tokens, max_depth, temperature,
                           seed, offset=0, without_replacement=False, b0=0):
        """Token-tree sampling verification (multi-round rejection); returns
        (accepted_len[B], out_tokens[B, max_depth+1], out_path[B, max_depth+1], flags[B])."""
        t, code, tsb, tsr = _logits(target)
        d, dcode, dsb, dsr = _logits(draft)
        B, N, V = t.shape
        if dcode != code or d.shape != (B, N, V):
            raise ValueError("draft logits must match the target's dtype and be [B, N, V]")
        par = np.ascontiguousarray(np.asarray(parent, dtype=np.int32).reshape(N))
        toks = np.ascontiguousarray(np.asarray(node_tokens, dtype=np.int32).reshape(B, N))
        W = max_depth + 1
        acc = np.zeros(B, np.int32)
        out = np.zeros((B, W), np.int32)
        path = np.zeros((B, W), np.int32)
        flags = np.zeros(B, np.int32)
        rc = self.lib.oracle_verify_tree_sample(_ptr(t), tsb, tsr, _ptr(d), dsb, dsr, code, B,
                                                int(b0), N, V, _ptr(par), _ptr(toks),
                                                int(max_depth), float(temperature),
                                                int(bool(without_replacement)), int(seed),
                                                int(offset), _ptr(acc), _ptr(out), _ptr(path),
                                                _ptr(flags))
        assert rc == 0
        return acc, out, path, flags

    def exact_probs_tree(self, t_logits, d_logits, parent, tokens, temperature,
                         without_replacement=False) -> np.ndarray:
        """Enumeration mode of the tree rule: P(final node = v, final token = j) as [N, V]."""
        t = np.ascontiguousarray(np.asarray(t_logits, dtype=np.float64))
        N, V = t.shape
        d = np.ascontiguousarray(np.asarray(d_logits, dtype=np.float64).reshape(N, V))
        par = np.ascontiguousarray(np.asarray(parent, dtype=np.int32).reshape(N))
        x = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32).reshape(N))
        prob = np.zeros((N, V), np.float64)
        rc = self.lib.oracle_exact_probs_tree(_ptr(t), _ptr(d), _ptr(par), _ptr(x), N, V,
                                              float(temperature), int(bool(without_replacement)),
                                              _ptr(prob))
        if rc != 0:
            raise ValueError("invalid tree, row or token")
        return prob


    def verify_typical(self, target, draft_tokens, temperature, epsilon, delta, seed, offset=0,
                       b0=0):
        """Typical acceptance; returns (accepted_len[B], out_tokens[B, gamma+1], flags[B],
        entropy[B, gamma+1] (H of each row the rule read, NaN elsewhere))."""
        t, code, tsb, tsr = _logits(target)
        B, G1, V = t.shape
        gamma = G1 - 1
        x = np.ascontiguousarray(np.asarray(draft_tokens, dtype=np.int32).reshape(B, gamma))
        acc = np.zeros(B, np.int32)
        out = np.zeros((B, G1), np.int32)
        flags = np.zeros(B, np.int32)
        H = np.zeros((B, G1), np.float64)
        rc = self.lib.oracle_verify_typical(_ptr(t), tsb, tsr, code, B, int(b0), gamma, V, _ptr(x),
                                            float(temperature), float(epsilon), float(delta),
                                            int(seed), int(offset), _ptr(acc), _ptr(out), _ptr(flags),
                                            _ptr(H))
        assert rc == 0
        return acc, out, flags, H

    def ngram_draft(self, history, lengths, n, k, pad):
        """Prompt-lookup drafts of a [B, T] int32 history with lengths[B]; returns
        (drafts [B, k] (-1 padded), counts [B])."""
        h = np.ascontiguousarray(np.asarray(history, dtype=np.int32))
        B, T = h.shape
        L = np.ascontiguousarray(np.asarray(lengths, dtype=np.int32).reshape(B))
        drafts = np.zeros((B, k), np.int32)
        count = np.zeros(B, np.int32)
        rc = self.lib.oracle_ngram_draft(_ptr(h), T, _ptr(L), B, int(n), int(k), int(bool(pad)),
                                         _ptr(drafts), _ptr(count))
        if rc != 0:
            raise ValueError("n must be >= 1 and k >= 0")
        return drafts, count


def philox4x32_10(ctr, key):
    return _load().philox4x32_10(ctr, key)


def uniform(seed, offset, b, i, purpose):
    return _load().uniform(seed, offset, b, i, purpose)


def row_stats(logits, temperature=1.0):
    return _load().row_stats(logits, temperature)


def verify_sample(target, draft, draft_tokens, temperature, seed, offset=0, b0=0,
                  diagnostics=False):
    return _load().verify_sample(target, draft, draft_tokens, temperature, seed, offset, b0,
                                 diagnostics)


def exact_probs(t_logits, d_logits, draft_tokens, temperature):
    return _load().exact_probs(t_logits, d_logits, draft_tokens, temperature)


def verify_greedy(target, draft_tokens):
    return _load().verify_greedy(target, draft_tokens)


def verify_tree_greedy(target, parent, node_tokens, max_depth):
    return _load().verify_tree_greedy(target, parent, node_tokens, max_depth)


def verify_tree_sample(target, draft, parent, node_tokens, max_depth, temperature, seed,
                       offset=0, without_replacement=False, b0=0):
    return _load().verify_tree_sample(target, draft, parent, node_tokens, max_depth, temperature,
                                      seed, offset, without_replacement, b0)


def exact_probs_tree(t_logits, d_logits, parent, tokens, temperature, without_replacement=False):
    return _load().exact_probs_tree(t_logits, d_logits, parent, tokens, temperature,
                                    without_replacement)


def verify_typical(target, draft_tokens, temperature, epsilon, delta, seed, offset=0, b0=0):
    return _load().verify_typical(target, draft_tokens, temperature, epsilon, delta, seed, offset, b0)


def ngram_draft(history, lengths, n, k, pad):
    return _load().ngram_draft(history, lengths, n, k, pad)


def default() -> Oracle:
    return _load()


def bf16_bits(t) -> np.ndarray:
    """Raw bf16 bit patterns of a CPU torch bf16 tensor as a uint16 numpy array."""
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def as_oracle_logits(t) -> np.ndarray:
    """A CPU view of a torch logits tensor in the form the oracle reads (fp32 or bf16 bits)."""
    import torch
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    return t.detach().cpu().contiguous().to(torch.float32).numpy()
