"""GPU parity of token-tree sampling verification (multi-round rejection) against the
oracle, through the C ABI.

Bar: accepted_len, every token and the path equal the oracle's, except on sequences the
oracle flags (a uniform within 1e-5 of an accept threshold or a CDF boundary, or a
near-zero residual); flagged and mismatched counts are recorded.  Over >= 10^4 sequences of
the B=64 workload, disagreements of any kind stay below 0.01 % (the walk's near-boundary
decisions are redone in double-float arithmetic).
"""
import numpy as np
import pytest
import torch

import speculative_decoding_verify_spec_gb300 as sv
from speculative_decoding_verify_spec_gb300 import binding
from speculative_decoding_verify_spec_gb300 import workloads as W

from parity_util import compare_tree_sample, host, oracle_tree_sample, record_rates

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _random_parent(rs, N):
    return [-1] + [int(rs.randint(0, v)) for v in range(1, N)]


def _run(s, label, offset=0, parent=None):
    par = s.parent if parent is None else parent
    acc, out, path = sv.spec_verify_tree_sample(s.target, s.draft, par, s.node_tokens, s.max_depth,
                                                s.temperature, s.seed, offset,
                                                without_replacement=s.without_replacement)
    o = oracle_tree_sample(s.target, s.draft, par, s.node_tokens, s.max_depth, s.temperature,
                           s.seed, offset, s.without_replacement)
    return compare_tree_sample(acc, out, path, *o, label=label)


CASES = [  # (tree, V, dtype, T, without_replacement)
    ("root", 1000, "fp32", 1.0, False),
    ("chain6", 777, "bf16", 0.8, False),
    ("random20", 777, "bf16", 1.0, True),
    ("random20", 4099, "fp32", 0.7, False),
    ("random40", 2048, "bf16", 1.3, True),
    ("shape64", 5000, "bf16", 1.0, True),
    ("shape64", 16385, "bf16", 1.0, False),
]


@pytest.mark.parametrize("tree,V,dtype,T,wor", CASES)
def test_small_trees_match_oracle(tree, V, dtype, T, wor):
    rs = np.random.RandomState(V + len(tree))
    parent = None
    if tree == "root":
        parent = [-1]
    elif tree == "chain6":
        parent = [-1, 0, 1, 2, 3, 4]
    elif tree.startswith("random"):
        parent = _random_parent(rs, int(tree[6:]))
    B = 48
    s = W.make_tree_sample(B, V, dtype, seed=V, verify_seed=17, device=DEV, N=64,
                           temperature=T, without_replacement=wor, parent=parent)
    # masked target logits: tokens the target never emits (p = 0)
    mask = torch.rand(s.target.shape, device=DEV, generator=torch.Generator(device=DEV).manual_seed(3)) < 0.05
    s.target.masked_fill_(mask, float("-inf"))
    for off in range(3):
        _run(s, f"tree sample {tree} V={V} {dtype} T={T} wor={wor}", offset=off)


def test_identical_rows_walk_the_first_children():
    # p = q at every node: every first child is accepted (u < 1), the walk ends at a leaf
    s = W.make_tree_sample(32, 3000, "bf16", seed=5, device=DEV, N=64, without_replacement=True)
    s.draft.copy_(s.target)
    acc, out, path = sv.spec_verify_tree_sample(s.target, s.draft, s.parent, s.node_tokens,
                                                s.max_depth, 1.0, 9)
    o = oracle_tree_sample(s.target, s.draft, s.parent, s.node_tokens, s.max_depth, 1.0, 9)
    compare_tree_sample(acc, out, path, *o, label="tree sample p = q")
    par = s.parent.cpu().tolist()
    first = [min([c for c in range(len(par)) if par[c] == v], default=-1) for v in range(len(par))]
    walk = [0]
    while first[walk[-1]] >= 0:
        walk.append(first[walk[-1]])
    assert (acc.cpu().numpy() == len(walk) - 1).all()
    assert (path.cpu().numpy()[:, :len(walk)] == np.array(walk)).all()


def test_bad_inputs_and_unread_rows():
    s = W.make_tree_sample(6, 1000, "fp32", seed=8, device=DEV, N=64, without_replacement=False)
    s.target[0, 0, 5] = float("nan")          # the root's target row
    s.draft[1, 0, :] = float("-inf")          # the root's draft row (the root has children)
    s.node_tokens[2, 7] = 1000                # a token out of range
    par = s.parent.cpu().tolist()
    leaves = [v for v in range(len(par)) if v not in par]
    s.draft[3, leaves] = float("nan")         # draft rows of leaves are never read
    acc, out, path = sv.spec_verify_tree_sample(s.target, s.draft, s.parent, s.node_tokens,
                                                s.max_depth, 1.0, 4)
    o = oracle_tree_sample(s.target, s.draft, s.parent, s.node_tokens, s.max_depth, 1.0, 4)
    compare_tree_sample(acc, out, path, *o, label="tree sample bad inputs")
    a = acc.cpu().numpy()
    assert (a[:3] == -1).all() and (a[3:] >= 0).all()
    # a malformed or too deep tree makes every sequence -1
    for bad_par, D in (([-1, 0, 2], 2), ([0, 0, 1], 2), ([-1, 0, 1], 1)):
        t = torch.zeros((2, 3, 50), device=DEV)
        acc, out, path = sv.spec_verify_tree_sample(t, t, torch.tensor(bad_par, dtype=torch.int32, device=DEV),
                                                    torch.zeros((2, 3), dtype=torch.int32, device=DEV), D,
                                                    1.0, 0)
        assert (acc == -1).all() and (out == -1).all() and (path == -1).all()


def test_unaligned_rows():
    # rows that start off a 16-byte boundary take the element-wise load path
    base = W.make_tree_sample(16, 3001, "bf16", seed=12, device=DEV, N=64, without_replacement=True)
    B, N, V = base.target.shape
    tbig = torch.zeros((B, N, V + 3), device=DEV, dtype=torch.bfloat16)
    dbig = torch.zeros((B, N, V + 3), device=DEV, dtype=torch.bfloat16)
    tbig[:, :, 1:V + 1] = base.target
    dbig[:, :, 1:V + 1] = base.draft
    t, d = tbig[:, :, 1:V + 1], dbig[:, :, 1:V + 1]
    acc, out, path = sv.spec_verify_tree_sample(t, d, base.parent, base.node_tokens, base.max_depth,
                                                1.0, 21, without_replacement=True)
    o = oracle_tree_sample(base.target, base.draft, base.parent, base.node_tokens, base.max_depth,
                           1.0, 21, 0, True)
    compare_tree_sample(acc, out, path, *o, label="tree sample unaligned rows")


def test_full_size_workload():
    s = W.make("tree_sample_b64", device=DEV)
    n = mism = flg = 0
    for off in range(4):
        a, b, c = _run(s, f"full tree_sample_b64 offset {off}", offset=off)
        n, mism, flg = n + a, mism + b, flg + c
    assert n == 256


def test_disagreements_are_below_one_in_ten_thousand():
    """160 rounds of the B=64 tree workload (fresh uniforms per round via the offset): every
    disagreement with the oracle is flagged, fewer than 0.01 % of the 10,240 sequences
    disagree at all, the re-walk ran and no grid barrier gave up."""
    s = W.make("tree_sample_b64", device=DEV)
    B, N, V = s.target.shape
    ws = torch.empty(sv.spec_verify_workspace_size(binding.MODE_TREE_SAMPLE, B, N, V, binding.BF16),
                     dtype=torch.uint8, device=DEV)
    t, d, x = host(s.target), host(s.draft), s.node_tokens.cpu().numpy()
    total = mism = flg = marked = redone = 0
    flags = []
    for off in range(1, 161):
        acc, out, path = sv.spec_verify_tree_sample(s.target, s.draft, s.parent, s.node_tokens, s.max_depth,
                                                    s.temperature, s.seed, off,
                                                    without_replacement=s.without_replacement, workspace=ws)
        m, r, status, marks = binding.call_status(ws, binding.MODE_TREE_SAMPLE, B, N, V, binding.BF16)
        assert status == 0 and m == int((marks != 0).sum()) and r == m
        marked, redone = marked + m, redone + r
        o = oracle_tree_sample(t, d, s.parent, x, s.max_depth, s.temperature, s.seed, off,
                               s.without_replacement)
        n, mm, f = compare_tree_sample(acc, out, path, *o, label=f"tree_sample_b64 offset {off}", record=False)
        total, mism, flg = total + n, mism + mm, flg + f
        flags.append(o[3])
    record_rates("tree_sample_b64 x160 rounds", total, mism, flg, np.concatenate(flags), redraw_marked=marked,
                 redraw_redone=redone)
    assert total == 10240
    assert marked > 0  # the re-walk is exercised
    assert mism < 1e-4 * total, (mism, total)



def test_wide_nodes_and_leaves_redo_every_final_draw():
    """A root with 12 children, one of them with 18 children, the others leaves; the draft far
    from the target, so most walks reject all 12 at the root.  A sequence marked only at its
    final draw is redone by the exponentials kernel's grid-wide passes at the root (up to 12
    rounds, several sequences in lock step), by the re-walk at the 18-child node (more
    children than that re-draw replays), and at a leaf the draw is from p alone.  Over 60
    rounds of 64 sequences every marked sequence is redone and equals the oracle, and each
    of the three kinds of final-only mark occurs."""
    parent = [-1] + [0] * 12 + [1] * 18
    s = W.make_tree_sample(64, 128256, "bf16", seed=4242, verify_seed=99, device=DEV, temperature=1.0,
                           without_replacement=True, parent=parent, draft_scale=0.3, noise_std=3.0)
    B, N, V = s.target.shape
    ws = torch.empty(sv.spec_verify_workspace_size(binding.MODE_TREE_SAMPLE, B, N, V, binding.BF16),
                     dtype=torch.uint8, device=DEV)
    t, d, x = host(s.target), host(s.draft), s.node_tokens.cpu().numpy()
    kinds = {"root": 0, "wide": 0, "leaf": 0}
    for off in range(60):
        acc, out, path = sv.spec_verify_tree_sample(s.target, s.draft, s.parent, s.node_tokens, s.max_depth,
                                                    s.temperature, s.seed, off,
                                                    without_replacement=s.without_replacement, workspace=ws)
        m, r, status, marks = binding.call_status(ws, binding.MODE_TREE_SAMPLE, B, N, V, binding.BF16)
        assert status == 0 and r == m == int((marks != 0).sum()), (off, m, r, status)
        o = oracle_tree_sample(t, d, s.parent, x, s.max_depth, s.temperature, s.seed, off, s.without_replacement)
        compare_tree_sample(acc, out, path, *o, label=f"wide tree offset {off}", record=False)
        a, op, pp = acc.cpu().numpy(), out.cpu().numpy(), path.cpu().numpy()
        for b in np.nonzero(marks)[0]:
            assert a[b] == o[0][b] and (op[b] == o[1][b]).all() and (pp[b] == o[2][b]).all(), (off, b)
            if marks[b] == 2:  # marked only at the final draw
                node = pp[b][a[b]]
                kinds["root" if node == 0 else "wide" if node == 1 else "leaf"] += 1
    print("final-only marks by the node they were drawn at:", kinds)
    assert min(kinds.values()) >= 1, kinds
