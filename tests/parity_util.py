"""Helpers shared by the GPU parity tests: run the oracle (in threads over sequence ranges)
on the same inputs the CUDA path sees, and compare."""
from __future__ import annotations

import json
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def host(t: torch.Tensor) -> np.ndarray:
    return oracle.as_oracle_logits(t)


def _ranges(B, parts):
    step = max(1, (B + parts - 1) // parts)
    return [(s, min(B, s + step)) for s in range(0, B, step)]


def oracle_sample(target, draft, tokens, T, seed, offset=0, threads=None, diagnostics=False):
    """The oracle over the whole batch, split over threads (each range keeps its global
    sequence index b0, which keys the uniforms).  Inputs may be CUDA tensors or the host
    arrays returned by host() (to convert once for many calls)."""
    # the C-ABI call receives the temperature as a float: the oracle divides by that value
    T = float(np.float32(T))
    t = target if isinstance(target, np.ndarray) else host(target)
    d = draft if isinstance(draft, np.ndarray) else host(draft)
    x = tokens if isinstance(tokens, np.ndarray) else tokens.cpu().numpy()
    x = x.astype(np.int32).reshape(t.shape[0], -1)
    B = t.shape[0]
    threads = threads or min(16, os.cpu_count() or 1)
    orc = oracle.default()

    def run(rg):
        s, e = rg
        return orc.verify_sample(t[s:e], d[s:e], x[s:e], T, seed, offset, b0=s,
                                 diagnostics=diagnostics)

    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(run, _ranges(B, threads)))
    return tuple(np.concatenate([p[i] for p in parts]) for i in range(4 if diagnostics else 3))


def oracle_greedy(target, tokens, threads=None):
    t = host(target)
    B = t.shape[0]
    x = tokens.cpu().numpy().astype(np.int32).reshape(B, -1)
    threads = threads or min(16, os.cpu_count() or 1)
    orc = oracle.default()
    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(lambda rg: orc.verify_greedy(t[rg[0]:rg[1]], x[rg[0]:rg[1]]),
                            _ranges(B, threads)))
    return tuple(np.concatenate([p[i] for p in parts]) for i in range(2))


def oracle_tree(target, parent, tokens, max_depth, threads=None):
    t = host(target)
    B = t.shape[0]
    par = np.asarray(parent.cpu().numpy() if torch.is_tensor(parent) else parent, np.int32)
    x = tokens.cpu().numpy().astype(np.int32)
    threads = threads or min(16, os.cpu_count() or 1)
    orc = oracle.default()
    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(lambda rg: orc.verify_tree_greedy(t[rg[0]:rg[1]], par, x[rg[0]:rg[1]],
                                                              max_depth), _ranges(B, threads)))
    return tuple(np.concatenate([p[i] for p in parts]) for i in range(4))


def oracle_tree_sample(target, draft, parent, tokens, max_depth, T, seed, offset=0,
                       without_replacement=False, threads=None):
    """The tree-sampling oracle over the whole batch, split over threads (global sequence
    index b0 keys the uniforms)."""
    T = float(np.float32(T))
    t = target if isinstance(target, np.ndarray) else host(target)
    d = draft if isinstance(draft, np.ndarray) else host(draft)
    B = t.shape[0]
    par = np.asarray(parent.cpu().numpy() if torch.is_tensor(parent) else parent, np.int32)
    x = tokens if isinstance(tokens, np.ndarray) else tokens.cpu().numpy()
    x = x.astype(np.int32).reshape(B, -1)
    threads = threads or min(16, os.cpu_count() or 1)
    orc = oracle.default()

    def run(rg):
        s, e = rg
        return orc.verify_tree_sample(t[s:e], d[s:e], par, x[s:e], max_depth, T, seed, offset,
                                      without_replacement, b0=s)

    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(run, _ranges(B, threads)))
    return tuple(np.concatenate([p[i] for p in parts]) for i in range(4))


def compare_tree_sample(acc, out, path, o_acc, o_out, o_path, o_flags, label="", record=True):
    """Lengths, tokens and paths must agree wherever the oracle raised no flag; returns
    (n, mismatches, flagged)."""
    acc, out, path = acc.cpu().numpy(), out.cpu().numpy(), path.cpu().numpy()
    same = (acc == o_acc) & (out == o_out).all(1) & (path == o_path).all(1)
    flagged = o_flags != 0
    bad = ~same & ~flagged
    if bad.any():
        i = int(np.nonzero(bad)[0][0])
        raise AssertionError(f"{label}: unflagged mismatch at sequence {i}: gpu acc={acc[i]} "
                             f"out={out[i].tolist()} path={path[i].tolist()} oracle acc={o_acc[i]} "
                             f"out={o_out[i].tolist()} path={o_path[i].tolist()}")
    n, mism, flg = len(acc), int((~same).sum()), int(flagged.sum())
    if record:
        record_rates(label, n, mism, flg, o_flags)
    return n, mism, flg


def compare_sample(acc, out, o_acc, o_out, o_flags, o_diag=None, label="", record=None):
    """Tokens and lengths must agree wherever the oracle raised no flag; returns
    (n, mismatches, flagged, diagnostics of the mismatched sequences)."""
    acc = acc.cpu().numpy()
    out = out.cpu().numpy()
    same = (acc == o_acc) & (out == o_out).all(1)
    flagged = o_flags != 0
    bad = ~same & ~flagged
    if bad.any():
        i = int(np.nonzero(bad)[0][0])
        extra = "" if o_diag is None else f" diag={o_diag[i].tolist()}"
        raise AssertionError(f"{label}: unflagged mismatch at sequence {i}: gpu acc={acc[i]} "
                             f"out={out[i].tolist()} oracle acc={o_acc[i]} out={o_out[i].tolist()}"
                             + extra)
    n, mism, flg = len(acc), int((~same).sum()), int(flagged.sum())
    mdiag = [] if o_diag is None else [
        {"mode": int(o_diag[i, 0]), "R": float(o_diag[i, 1]), "cdf_margin": float(o_diag[i, 2]),
         "accept_margin": float(o_diag[i, 3]), "acc_equal": bool(acc[i] == o_acc[i])}
        for i in np.nonzero(~same)[0]]
    if record is not None:
        record_rates(label, n, mism, flg, o_flags, mdiag)
    return n, mism, flg, mdiag


def record_rates(label, n, mismatches, flagged, flags, mismatch_diag=(), **extra):
    """Append the flag / mismatch counts of a parity case, as one JSON line, to the file that
    the SV_PARITY_LOG environment variable names (nothing is kept when it is unset)."""
    path = os.environ.get("SV_PARITY_LOG")
    if not path:
        return
    if os.path.dirname(path):
        os.makedirs(os.path.dirname(path), exist_ok=True)
    rec = {"case": label, "sequences": n, "mismatches": mismatches, "flagged": flagged,
           "flag_accept": int(((flags & 1) != 0).sum()), "flag_cdf": int(((flags & 2) != 0).sum()),
           "flag_residual_small": int(((flags & 4) != 0).sum()),
           "mismatch_diagnostics": list(mismatch_diag)[:50], **extra}
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")
