"""The seeded input generators: shapes, determinism and the pruned tree shape (CPU)."""
import collections

import torch

from speculative_decoding_verify_spec_gb300 import workloads as W


def test_sample_inputs_shapes_and_determinism():
    a = W.make("sample_b64", B=3, V=500)
    b = W.make("sample_b64", B=3, V=500)
    assert a.target.shape == (3, 6, 500) and a.draft.shape == (3, 5, 500)
    assert a.target.dtype == torch.bfloat16 and a.draft_tokens.dtype == torch.int32
    assert torch.equal(a.target, b.target) and torch.equal(a.draft_tokens, b.draft_tokens)
    assert ((a.draft_tokens >= 0) & (a.draft_tokens < 500)).all()
    c = W.make("sample_b1")
    assert c.target.dtype == torch.float32 and c.target.shape == (1, 5, 1000)


def test_peaked_rows_fraction():
    # with V = 50 an unboosted N(0, 3^2) row almost never exceeds 11.5
    s = W.make("sample_b256", B=200, V=50)
    rows = s.target.float().view(-1, 50)
    peaked = (rows.max(-1).values > 11.5).float().mean().item()
    assert 0.02 < peaked < 0.09


def test_greedy_drafts_match_argmax_mostly():
    g = W.make("greedy_b512", B=200, V=300)
    a = torch.argmax(g.target[:, :6].float(), -1)
    frac = (a == g.draft_tokens).float().mean().item()
    assert 0.7 < frac < 0.9


def test_tree_shape_counts():
    parent, depth = W.tree_shape((4, 3, 2, 2, 1, 1), 64)
    assert len(parent) == 64 and parent[0] == -1
    assert all(0 <= parent[v] < v for v in range(1, 64))
    assert [collections.Counter(depth)[d] for d in range(7)] == [1, 4, 9, 11, 13, 13, 13]
    t = W.make("tree_b64", B=4, V=100)
    assert t.target.shape == (4, 64, 100) and t.max_depth == 6


def test_logical_bytes_formula():
    assert W.logical_bytes("sample_b256") == 256 * 17 * 128256 * 2 + 4 * 256 * 8 + 4 * 256 * 10
    assert W.logical_bytes("greedy_b512") == 512 * 7 * 152064 * 2 + 4 * 512 * 6 + 4 * 512 * 8
