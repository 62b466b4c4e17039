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


def test_metric_bytes_match_the_printed_sizes():
    # the metric's bytes: every logit once plus the small integer inputs and outputs,
    # against the sizes printed beside the five workloads (to their last printed digit)
    assert W.logical_bytes("sample_b1") == 1 * 9 * 1000 * 4 + 4 * 4 + 4 * 6
    assert abs(W.logical_bytes("sample_b64") / 1e6 - 45.06) < 0.01
    assert abs(W.logical_bytes("sample_b256") / 1e9 - 1.1163) < 1e-4
    assert abs(W.logical_bytes("greedy_b512") / 1e9 - 1.0900) < 1e-4
    assert abs(W.logical_bytes("tree_b64") / 1e9 - 1.0507) < 1e-4


def test_rows_and_target_only_bytes():
    assert W.rows("sample_b256") == 256 * 17
    assert W.rows("typical_b256") == W.rows("onehot_b256") == 256 * 9     # no draft rows
    assert W.rows("greedy_b512") == 512 * 7 and W.rows("tree_b64") == 64 * 64
    assert W.logical_bytes("typical_b256") == 256 * 9 * 128256 * 2 + 4 * 256 * 8 + 4 * 256 * 10
    assert W.logical_bytes("onehot_b256") == W.logical_bytes("typical_b256")
    assert W.logical_bytes("ngram_b256") == 256 * (16384 * 4 + 4 + 8 * 4 + 4)


def test_tree_sample_children_are_distinct_draws():
    s = W.make("tree_sample_b64", B=6, V=40)
    par = s.parent.tolist()
    assert s.target.shape == (6, 64, 40) and s.draft.shape == (6, 64, 40)
    assert s.without_replacement and s.max_depth == 6
    for v in range(64):
        kids = [c for c in range(1, 64) if par[c] == v]
        if len(kids) > 1:  # without replacement: siblings carry distinct tokens
            toks = s.node_tokens[:, kids]
            for b in range(6):
                assert len(set(toks[b].tolist())) == len(kids)
    assert ((s.node_tokens[:, 1:] >= 0) & (s.node_tokens[:, 1:] < 40)).all()


def test_ngram_histories_are_ragged_and_copy_heavy():
    g = W.make("ngram_b256", B=16, T=4096)
    L = g.lengths
    assert g.history.shape == (16, 4096) and g.history.dtype == torch.int32
    assert ((L >= 4096 - 1024) & (L <= 4096)).all() and len(set(L.tolist())) > 1
    assert ((g.history >= 0) & (g.history < 128256)).all()
    # most tails have an earlier occurrence (the last span repeats earlier text w.p. 0.8)
    hits = 0
    for b in range(16):
        h, n = g.history[b, :int(L[b])].tolist(), g.n
        tail = h[-n:]
        hits += any(h[i:i + n] == tail for i in range(len(h) - n))
    assert hits >= 8
