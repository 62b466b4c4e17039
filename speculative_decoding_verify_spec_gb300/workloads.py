"""Seeded synthetic inputs for the verification step.

This module is shared by the tests, the bench and the smoke check, and feeds the CUDA
library and the oracle alike.  It holds none of the verification arithmetic: it only draws
logits, drafts and trees with the shapes and value distributions of the five workloads
below, from a seeded ``torch.Generator`` on the requested device.

Draft tokens are a *drafter's* output, so simulating them needs a draw from the draft
distribution (Gumbel-max over ``draft / T``) or the target argmax (``torch.argmax``, which
returns the first maximal index); both are library calls standing in for a drafter, and
neither side of a parity check relies on how the drafts were made.

Workloads (vocabulary sizes, draft lengths and distributions as specified for the bench):
  sample_b1      sampling, B=1,   V=1000,   gamma=4, fp32, t ~ N(0,2^2), d = t + N(0,0.5^2), T=1
  sample_b64     sampling, B=64,  V=32000,  gamma=5, bf16, t ~ N(0,3^2) + Zipf(1.1) boost on a
                 random vocabulary permutation, d = t + N(0,1), T=1
  sample_b256    sampling, B=256, V=128256, gamma=8, bf16, t ~ N(0,3^2) with 5% of rows peaked
                 (one random token +12), d = 0.8 t + N(0,1), T=0.7 on both
  greedy_b512    greedy,   B=512, V=152064, gamma=6, bf16, t ~ N(0,2^2), draft_i = argmax row i
                 w.p. 0.8 else uniform
  tree_b64       tree,     B=64,  N=64 nodes (depth 6, fanouts 4,3,2,2,1,1 pruned to 64 nodes),
                 V=128256, bf16, t ~ N(0,2^2); per internal node one random child carries the
                 parent's argmax w.p. 0.7, every other child a uniform token
  tree_sample_b64  token-tree sampling (multi-round rejection) on the same tree, B=64,
                 V=128256, bf16, t ~ N(0,2^2) at every node, d = 0.8 t + N(0,1), T=1; every
                 internal node's children are a drafter's draws from softmax(d_v / T) without
                 replacement (Gumbel top-k, in draw order)
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

WORKLOADS = {
    "sample_b1": dict(mode="sample", B=1, gamma=4, V=1000, dtype="fp32", temperature=1.0,
                      input_seed=1001, verify_seed=0),
    "sample_b64": dict(mode="sample", B=64, gamma=5, V=32000, dtype="bf16", temperature=1.0,
                       input_seed=1002, verify_seed=0x5EED + 2),
    "sample_b256": dict(mode="sample", B=256, gamma=8, V=128256, dtype="bf16", temperature=0.7,
                        input_seed=1003, verify_seed=0x5EED + 3),
    "greedy_b512": dict(mode="greedy", B=512, gamma=6, V=152064, dtype="bf16", input_seed=1004),
    "tree_b64": dict(mode="tree", B=64, N=64, V=128256, dtype="bf16", input_seed=1005,
                     branching=(4, 3, 2, 2, 1, 1)),
    "tree_sample_b64": dict(mode="tree_sample", B=64, N=64, V=128256, dtype="bf16",
                            input_seed=1006, verify_seed=0x5EED + 6, temperature=1.0,
                            branching=(4, 3, 2, 2, 1, 1), without_replacement=True),
}
WORKLOADS["ngram_b256"] = dict(mode="ngram", B=256, T=16384, V=128256, n=3, k=8, pad=False, input_seed=1007)
# the same inputs, verified by the lazy entries (rows read only where the rule needs them)
for _base in ("sample_b256", "greedy_b512", "tree_b64"):
    WORKLOADS[_base + "_lazy"] = dict(WORKLOADS[_base], lazy=True, base=_base)
# the B=256 sampling inputs under typical acceptance (target rows only; the threshold's
# constants are workload parameters chosen for a mid-range acceptance -- the pages give none)
WORKLOADS["typical_b256"] = dict(WORKLOADS["sample_b256"], typical=True, base="sample_b256", epsilon=0.1, delta=0.3)
# ... and verified by sampling against a one-hot q (a prompt-lookup drafter's): target rows only
WORKLOADS["onehot_b256"] = dict(WORKLOADS["sample_b256"], onehot=True, base="sample_b256")

DESCRIPTIONS = {
    "sample_b1": "sampling verify B=1 V=1000 gamma=4 fp32 T=1.0",
    "sample_b64": "sampling verify B=64 V=32000 gamma=5 bf16 T=1.0 (Zipf-boosted target)",
    "sample_b256": "sampling verify B=256 V=128256 gamma=8 bf16 T=0.7 (5% peaked rows)",
    "greedy_b512": "greedy verify B=512 V=152064 gamma=6 bf16",
    "tree_b64": "greedy token-tree verify B=64 N=64 depth=6 V=128256 bf16",
    "tree_sample_b64": ("token-tree sampling verify (multi-round rejection) B=64 N=64 depth=6 "
                        "V=128256 bf16 T=1.0, children drawn from q without replacement"),
}
DESCRIPTIONS["ngram_b256"] = ("prompt-lookup drafting B=256 histories of up to 16384 tokens (V=128256, copy-heavy), "
                              "n=3, k=8")
for _base in ("sample_b256", "greedy_b512", "tree_b64"):
    DESCRIPTIONS[_base + "_lazy"] = DESCRIPTIONS[_base] + ", lazy (rows read only where the rule needs them)"
DESCRIPTIONS["typical_b256"] = ("typical acceptance B=256 V=128256 gamma=8 bf16 T=0.7, threshold "
                                "min(0.1, 0.3 exp(-H)), the sampling workload's target rows and drafts")
DESCRIPTIONS["onehot_b256"] = ("sampling verify against a one-hot q B=256 V=128256 gamma=8 bf16 T=0.7, "
                               "the sampling workload's target rows and drafts")


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def _randn(shape, g, device, std=1.0):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def _round(x: torch.Tensor, dtype: str) -> torch.Tensor:
    return x.to(torch.bfloat16) if dtype == "bf16" else x.to(torch.float32)


def _gumbel_draw(logits_over_T: torch.Tensor, g, device) -> torch.Tensor:
    """One draw per row from softmax(logits_over_T) by the Gumbel-max trick (a drafter)."""
    u = torch.rand(logits_over_T.shape, generator=g, device=device, dtype=torch.float32)
    u = u.clamp_(min=1e-20, max=1.0 - 1e-7)
    gumbel = -torch.log(-torch.log(u))
    return torch.argmax(logits_over_T + gumbel, dim=-1).to(torch.int32)


@dataclass
class SampleInputs:
    target: torch.Tensor        # [B, gamma+1, V]
    draft: torch.Tensor         # [B, gamma, V]
    draft_tokens: torch.Tensor  # [B, gamma] int32
    temperature: float
    seed: int
    offset: int = 0


@dataclass
class GreedyInputs:
    target: torch.Tensor        # [B, gamma+1, V]
    draft_tokens: torch.Tensor  # [B, gamma] int32


@dataclass
class TreeInputs:
    target: torch.Tensor        # [B, N, V]
    parent: torch.Tensor        # [N] int32
    node_tokens: torch.Tensor   # [B, N] int32
    max_depth: int
    depth: list = field(default_factory=list)


def make_sample(B, gamma, V, dtype="bf16", recipe="normal", temperature=1.0, seed=1,
                verify_seed=0, device="cpu", target_std=None, noise_std=None,
                draft_scale=None, peaked_frac=None, peak_boost=12.0, zipf_s=None):
    """Sampling-verify inputs.

    recipe "normal":  t ~ N(0, target_std^2), d = draft_scale * t + N(0, noise_std^2)
    recipe "zipf":    t ~ N(0, target_std^2) - zipf_s * ln(rank_pi(j) + 1) for a random
                      permutation pi of the vocabulary (fixed per call)
    recipe "peaked":  like "normal", then a fraction peaked_frac of target rows gets one
                      uniformly chosen token raised by peak_boost (before the draft is made)
    """
    g = _gen(seed, device)
    target_std = 2.0 if target_std is None else target_std
    noise_std = 0.5 if noise_std is None else noise_std
    draft_scale = 1.0 if draft_scale is None else draft_scale
    t = _randn((B, gamma + 1, V), g, device, target_std)
    if recipe == "zipf":
        s = 1.1 if zipf_s is None else zipf_s
        perm = torch.randperm(V, generator=g, device=device)
        rank = torch.empty(V, dtype=torch.float32, device=device)
        rank[perm] = torch.arange(V, dtype=torch.float32, device=device)
        t = t - s * torch.log(rank + 1.0)
    elif recipe == "peaked":
        frac = 0.05 if peaked_frac is None else peaked_frac
        rows = t.view(-1, V)
        chosen = torch.rand(rows.shape[0], generator=g, device=device) < frac
        tok = torch.randint(0, V, (rows.shape[0],), generator=g, device=device)
        idx = torch.nonzero(chosen).flatten()
        rows[idx, tok[idx]] += peak_boost
    elif recipe != "normal":
        raise ValueError(recipe)
    d = draft_scale * t[:, :gamma, :] + _randn((B, gamma, V), g, device, noise_std)
    t_r = _round(t, dtype)
    d_r = _round(d, dtype)
    if gamma > 0:
        x = _gumbel_draw(d_r.float() / temperature, g, device)
    else:
        x = torch.zeros((B, 0), dtype=torch.int32, device=device)
    return SampleInputs(t_r.contiguous(), d_r.contiguous(), x.contiguous(), float(temperature),
                        int(verify_seed))


def make_greedy(B, gamma, V, dtype="bf16", seed=1, device="cpu", target_std=2.0, p_match=0.8):
    """Greedy-verify inputs: t ~ N(0, target_std^2); draft_i = argmax(row i) w.p. p_match."""
    g = _gen(seed, device)
    t = _round(_randn((B, gamma + 1, V), g, device, target_std), dtype)
    a = torch.argmax(t[:, :gamma, :].float(), dim=-1).to(torch.int32)
    rnd = torch.randint(0, V, (B, gamma), generator=g, device=device, dtype=torch.int32)
    keep = torch.rand((B, gamma), generator=g, device=device) < p_match
    x = torch.where(keep, a, rnd)
    return GreedyInputs(t.contiguous(), x.contiguous())


def tree_shape(branching=(4, 3, 2, 2, 1, 1), n_nodes=64):
    """The pruned token tree: parent[] in BFS order (parent before child) and depths.

    The full tree with these per-depth fanouts has more nodes than the budget, so the
    n_nodes nodes with the smallest (sum of sibling ranks along the root path, BFS index)
    are kept -- the most-likely-path-first shape of top-k draft trees.  That set contains
    every kept node's parent, and renumbering it in BFS order keeps parent[i] < i.
    """
    nodes = [(0, -1, 0, 0)]  # (bfs index, parent bfs index, depth, rank sum)
    frontier = [0]
    for depth, fan in enumerate(branching, start=1):
        nxt = []
        for par in frontier:
            for rank in range(fan):
                idx = len(nodes)
                nodes.append((idx, par, depth, nodes[par][3] + rank))
                nxt.append(idx)
        frontier = nxt
    kept = sorted(nodes, key=lambda n: (n[3], n[0]))[:n_nodes]
    kept_ids = sorted(n[0] for n in kept)
    renum = {old: new for new, old in enumerate(kept_ids)}
    parent = [-1] * len(kept_ids)
    depth = [0] * len(kept_ids)
    for old in kept_ids:
        _, par, dep, _ = nodes[old]
        parent[renum[old]] = -1 if par < 0 else renum[par]
        depth[renum[old]] = dep
    return parent, depth


def make_tree(B, V, dtype="bf16", seed=1, device="cpu", branching=(4, 3, 2, 2, 1, 1), N=64,
              target_std=2.0, p_match=0.7, parent=None):
    """Tree-verify inputs on the pruned tree (or a given parent list)."""
    if parent is None:
        parent, depth = tree_shape(branching, N)
    else:
        depth = [0] * len(parent)
        for v in range(1, len(parent)):
            depth[v] = depth[parent[v]] + 1
    N = len(parent)
    g = _gen(seed, device)
    t = _round(_randn((B, N, V), g, device, target_std), dtype)
    a = torch.argmax(t.float(), dim=-1).to(torch.int32)  # [B, N]
    tokens = torch.randint(0, V, (B, N), generator=g, device=device, dtype=torch.int32)
    children = [[] for _ in range(N)]
    for v in range(1, N):
        children[parent[v]].append(v)
    internal = [v for v in range(N) if children[v]]
    if internal:
        pick_u = torch.rand((B, len(internal)), generator=g, device=device).cpu()
        do_u = torch.rand((B, len(internal)), generator=g, device=device).cpu()
        rows, cols, srcs = [], [], []
        for k, v in enumerate(internal):
            ch = children[v]
            for b in range(B):
                if float(do_u[b, k]) < p_match:
                    c = ch[min(int(float(pick_u[b, k]) * len(ch)), len(ch) - 1)]
                    rows.append(b)
                    cols.append(c)
                    srcs.append(v)
        if rows:
            r = torch.tensor(rows, device=device, dtype=torch.long)
            c = torch.tensor(cols, device=device, dtype=torch.long)
            s = torch.tensor(srcs, device=device, dtype=torch.long)
            tokens[r, c] = a[r, s]
    par_t = torch.tensor(parent, dtype=torch.int32, device=device)
    return TreeInputs(t.contiguous(), par_t, tokens.contiguous(), max(depth), list(depth))


@dataclass
class TreeSampleInputs:
    target: torch.Tensor        # [B, N, V]
    draft: torch.Tensor         # [B, N, V]
    parent: torch.Tensor        # [N] int32
    node_tokens: torch.Tensor   # [B, N] int32
    max_depth: int
    temperature: float
    seed: int
    without_replacement: bool
    depth: list = field(default_factory=list)


def draw_children(draft_over_T: torch.Tensor, k: int, without_replacement: bool, g, device):
    """k ordered children per row drawn from softmax(draft_over_T) ([rows, k] int32): a
    drafter's draws, by Gumbel-max (with replacement, k independent draws) or Gumbel
    top-k (without replacement: the keys sorted descending give the draw order)."""
    if not without_replacement:
        return torch.stack([_gumbel_draw(draft_over_T, g, device) for _ in range(k)], dim=-1)
    u = torch.rand(draft_over_T.shape, generator=g, device=device, dtype=torch.float32)
    u = u.clamp_(min=1e-20, max=1.0 - 1e-7)
    keys = draft_over_T + (-torch.log(-torch.log(u)))
    return torch.topk(keys, k, dim=-1, sorted=True).indices.to(torch.int32)


def make_tree_sample(B, V, dtype="bf16", seed=1, verify_seed=0, device="cpu",
                     branching=(4, 3, 2, 2, 1, 1), N=64, temperature=1.0,
                     without_replacement=True, target_std=2.0, draft_scale=0.8, noise_std=1.0,
                     parent=None):
    """Tree-sampling inputs: target and draft logits at every node of the pruned tree (or a
    given parent list), every internal node's children drawn from q at that node."""
    if parent is None:
        parent, depth = tree_shape(branching, N)
    else:
        depth = [0] * len(parent)
        for v in range(1, len(parent)):
            depth[v] = depth[parent[v]] + 1
    N = len(parent)
    g = _gen(seed, device)
    t32 = _randn((B, N, V), g, device, target_std)
    d32 = draft_scale * t32 + _randn((B, N, V), g, device, noise_std)
    t, d = _round(t32, dtype), _round(d32, dtype)
    del t32, d32
    tokens = torch.zeros((B, N), device=device, dtype=torch.int32)
    children = [[] for _ in range(N)]
    for v in range(1, N):
        children[parent[v]].append(v)
    for v in range(N):
        if children[v]:
            drawn = draw_children(d[:, v].float() / temperature, len(children[v]),
                                  without_replacement, g, device)
            tokens[:, children[v]] = drawn
    par_t = torch.tensor(parent, dtype=torch.int32, device=device)
    return TreeSampleInputs(t.contiguous(), d.contiguous(), par_t, tokens.contiguous(),
                            max(depth), float(temperature), int(verify_seed),
                            bool(without_replacement), list(depth))


@dataclass
class NgramInputs:
    history: torch.Tensor   # [B, T] int32
    lengths: torch.Tensor   # [B] int32
    n: int
    k: int
    pad: bool


def make_ngram(B, T, V, n=3, k=8, pad=False, seed=1, device="cpu", copies=64, span=(16, 64),
               tail_copy=0.8):
    """Copy-heavy token histories: uniform tokens into which `copies` spans of earlier text
    are copied (the repetition prompt lookup exploits); with probability tail_copy the last
    span of a history repeats an earlier one, so its tail usually has an earlier occurrence.
    Lengths are ragged in [T - 1024, T]."""
    import numpy as np
    rs = np.random.RandomState(seed)
    h = rs.randint(0, V, (B, T)).astype(np.int32)
    lengths = (T - rs.randint(0, min(1024, T), B)).astype(np.int32)
    for b in range(B):
        L = int(lengths[b])
        for _ in range(copies):
            ln = int(rs.randint(span[0], span[1] + 1))
            if L <= 2 * ln + 1:
                break
            dst = int(rs.randint(ln, L - ln))
            src = int(rs.randint(0, dst - ln + 1))
            h[b, dst:dst + ln] = h[b, src:src + ln]
        if rs.rand() < tail_copy and L > 2 * span[1] + 1:
            ln = span[1]
            src = int(rs.randint(0, L - 2 * ln))
            h[b, L - ln:L] = h[b, src:src + ln]
    return NgramInputs(torch.from_numpy(h).to(device), torch.from_numpy(lengths).to(device), n, k, pad)


def make(name: str, device="cpu", **overrides):
    """Inputs of a named workload (shapes may be overridden to make a smaller case)."""
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    name = cfg.get("base", name)
    mode = cfg["mode"]
    if mode == "sample":
        common = dict(B=cfg["B"], gamma=cfg["gamma"], V=cfg["V"], dtype=cfg["dtype"],
                      temperature=cfg["temperature"], seed=cfg["input_seed"],
                      verify_seed=cfg["verify_seed"], device=device)
        if name == "sample_b1":
            return make_sample(recipe="normal", target_std=2.0, noise_std=0.5, **common)
        if name == "sample_b64":
            return make_sample(recipe="zipf", target_std=3.0, noise_std=1.0, zipf_s=1.1, **common)
        return make_sample(recipe="peaked", target_std=3.0, noise_std=1.0, draft_scale=0.8,
                           peaked_frac=0.05, peak_boost=12.0, **common)
    if mode == "greedy":
        return make_greedy(cfg["B"], cfg["gamma"], cfg["V"], cfg["dtype"], cfg["input_seed"],
                           device)
    if mode == "ngram":
        return make_ngram(cfg["B"], cfg["T"], cfg["V"], cfg["n"], cfg["k"], cfg["pad"], cfg["input_seed"], device)
    if mode == "tree_sample":
        return make_tree_sample(cfg["B"], cfg["V"], cfg["dtype"], cfg["input_seed"],
                                cfg["verify_seed"], device, tuple(cfg["branching"]), cfg["N"],
                                cfg["temperature"], cfg["without_replacement"])
    return make_tree(cfg["B"], cfg["V"], cfg["dtype"], cfg["input_seed"], device,
                     tuple(cfg["branching"]), cfg["N"])


def logical_bytes(name: str, **overrides) -> int:
    """Bytes the metric counts for one verify call: every logit once plus the small
    integer inputs and outputs (for the drafter: every history token once, and the drafts)."""
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    if cfg["mode"] == "ngram":
        return cfg["B"] * (cfg["T"] * 4 + 4 + cfg["k"] * 4 + 4)
    s = 2 if cfg["dtype"] == "bf16" else 4
    B, V = cfg["B"], cfg["V"]
    if cfg["mode"] == "sample" and (cfg.get("typical") or cfg.get("onehot")):  # target rows only
        g = cfg["gamma"]
        return B * (g + 1) * V * s + 4 * B * g + 4 * B * (g + 2)
    if cfg["mode"] == "sample":
        g = cfg["gamma"]
        return B * (2 * g + 1) * V * s + 4 * B * g + 4 * B * (g + 2)
    if cfg["mode"] == "greedy":
        g = cfg["gamma"]
        return B * (g + 1) * V * s + 4 * B * g + 4 * B * (g + 2)
    N = cfg["N"]
    _, depth = tree_shape(tuple(cfg["branching"]), N)
    D = max(depth)
    if cfg["mode"] == "tree_sample":  # every target row and the draft rows of internal nodes
        internal = len(set(tree_shape(tuple(cfg["branching"]), N)[0][1:]))
        return B * (N + internal) * V * s + 4 * B * N + 4 * N + 4 * B * (2 * D + 3)
    return B * N * V * s + 4 * B * N + 4 * N + 4 * B * (2 * D + 3)


def units(name: str, **overrides) -> int:
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    return cfg["B"]


def rows(name: str, **overrides) -> int:
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    if cfg["mode"] == "ngram":
        return cfg["B"]
    if cfg["mode"] == "sample":
        return cfg["B"] * ((1 if cfg.get("typical") or cfg.get("onehot") else 2) * cfg["gamma"] + 1)
    if cfg["mode"] == "greedy":
        return cfg["B"] * (cfg["gamma"] + 1)
    return cfg["B"] * cfg["N"]
