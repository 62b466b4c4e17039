"""GPU parity of greedy and greedy-tree verification against the oracle, through the C
ABI.  Bar: bit-exact accepted_len, tokens and paths (argmax ties to the lowest index)."""
import numpy as np
import pytest
import torch

import speculative_decoding_verify_spec_gb300 as sv
from speculative_decoding_verify_spec_gb300 import workloads as W

from parity_util import oracle_greedy, oracle_tree

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _eq(a, b):
    return np.array_equal(a.cpu().numpy() if torch.is_tensor(a) else a, b)


def _ties(B, R, V, dtype, seed, lo=-3, hi=4):
    """Small-integer logits: exact ties everywhere, so the lowest-index rule decides."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randint(lo, hi, (B, R, V), generator=g, device=DEV).float()
    return x.to(torch.bfloat16 if dtype == "bf16" else torch.float32)


@pytest.mark.parametrize("B,gamma,V,dtype", [(64, 6, 1, "bf16"), (64, 4, 5, "fp32"),
                                             (50, 6, 1000, "bf16"), (33, 3, 16385, "bf16"),
                                             (20, 7, 33000, "fp32"), (9, 0, 4000, "bf16"),
                                             (4, 40, 600, "bf16")])
def test_greedy_small_with_ties(B, gamma, V, dtype):
    t = _ties(B, gamma + 1, V, dtype, B + V)
    a = torch.argmax(t[:, :gamma].float(), -1).to(torch.int32)
    g = torch.Generator(device=DEV).manual_seed(7)
    rnd = torch.randint(0, V, (B, gamma), generator=g, device=DEV, dtype=torch.int32)
    x = torch.where(torch.rand((B, gamma), generator=g, device=DEV) < 0.8, a, rnd)
    acc, out = sv.spec_verify_greedy(t, x)
    o_acc, o_out = oracle_greedy(t, x)
    assert _eq(acc, o_acc) and _eq(out, o_out)


def test_greedy_bad_sequences_and_special_values():
    B, gamma, V = 10, 3, 20000
    t = _ties(B, gamma + 1, V, "bf16", 1)
    t[1, 2, 19999] = float("nan")
    t[2, 0, :] = float("-inf")                      # valid: argmax of an all -inf row is 0
    t[3, 1, 12345] = float("inf")                   # valid: +inf is the maximum
    t[4, 0, 5] = float("inf")
    t[4, 0, 6] = float("inf")
    x = torch.zeros((B, gamma), dtype=torch.int32, device=DEV)
    x[5, 2] = V
    x[6, 0] = -7
    acc, out = sv.spec_verify_greedy(t, x)
    o_acc, o_out = oracle_greedy(t, x)
    assert _eq(acc, o_acc) and _eq(out, o_out)
    assert (o_acc[[1, 5, 6]] == -1).all() and o_out[3, 1] in (-1, 12345)


def test_greedy_unaligned_and_strided():
    B, gamma, V = 16, 5, 30001
    base = _ties(B, gamma + 1, V + 3, "bf16", 4)
    t = base[:, :, 3:]                                 # misaligned by 6 bytes
    x = torch.argmax(t[:, :gamma].float(), -1).to(torch.int32)
    x[::3, 2] = 0
    acc, out = sv.spec_verify_greedy(t, x)
    o_acc, o_out = oracle_greedy(t.contiguous(), x)
    assert _eq(acc, o_acc) and _eq(out, o_out)


def test_greedy_full_size():
    g = W.make("greedy_b512", device=DEV)
    acc, out = sv.spec_verify_greedy(g.target, g.draft_tokens)
    o_acc, o_out = oracle_greedy(g.target, g.draft_tokens)
    assert _eq(acc, o_acc) and _eq(out, o_out)
    del g
    torch.cuda.empty_cache()


def _random_tree(rs, N):
    return [-1] + [int(rs.randint(0, v)) for v in range(1, N)]


@pytest.mark.parametrize("N,V,dtype", [(1, 100, "bf16"), (2, 3, "fp32"), (9, 5, "bf16"),
                                       (64, 20000, "bf16"), (200, 700, "fp32"), (1024, 64, "bf16")])
def test_tree_small(N, V, dtype):
    rs = np.random.RandomState(N * 7 + V)
    parent = _random_tree(rs, N)
    depth = [0] * N
    for v in range(1, N):
        depth[v] = depth[parent[v]] + 1
    B = 24
    t = _ties(B, N, V, dtype, N + V, lo=-2, hi=3)
    a = torch.argmax(t.float(), -1).cpu().numpy()
    tok = rs.randint(0, V, (B, N)).astype(np.int32)
    for b in range(B):
        for v in range(1, N):
            if rs.rand() < 0.7:
                tok[b, v] = a[b, parent[v]]
    par_t = torch.tensor(parent, dtype=torch.int32, device=DEV)
    tok_t = torch.tensor(tok, device=DEV)
    D = max(depth)
    acc, out, path = sv.spec_verify_tree_greedy(t, par_t, tok_t, D)
    o_acc, o_out, o_path, _ = oracle_tree(t, parent, tok_t, D)
    assert _eq(acc, o_acc) and _eq(out, o_out) and _eq(path, o_path)
    # wider outputs than needed are padded with -1
    acc2, out2, path2 = sv.spec_verify_tree_greedy(t, par_t, tok_t, min(N - 1, D + 2), with_path=False)
    assert path2 is None and _eq(acc2, o_acc)
    assert _eq(out2[:, :D + 1], o_out) and (out2[:, D + 1:] == -1).all()


def test_tree_invalid_or_too_deep():
    B, N, V = 3, 5, 50
    t = _ties(B, N, V, "bf16", 9)
    tok = torch.zeros((B, N), dtype=torch.int32, device=DEV)
    for parent, D in (([-1, 0, 3, 1, 1], 3), ([0, 0, 1, 2, 3], 3), ([-1, 0, 1, 2, 3], 2)):
        acc, out, path = sv.spec_verify_tree_greedy(t, torch.tensor(parent, dtype=torch.int32, device=DEV),
                                                    tok, D)
        assert (acc == -1).all() and (out == -1).all() and (path == -1).all()
    tok[1, 3] = V + 1
    t[2, 4, 0] = float("nan")
    acc, out, path = sv.spec_verify_tree_greedy(t, torch.tensor([-1, 0, 0, 1, 2], dtype=torch.int32,
                                                                device=DEV), tok, 2)
    o_acc, o_out, o_path, _ = oracle_tree(t, [-1, 0, 0, 1, 2], tok, 2)
    assert _eq(acc, o_acc) and _eq(out, o_out) and _eq(path, o_path)
    assert o_acc[1] == -1 and o_acc[2] == -1 and o_acc[0] >= 0


def test_chain_tree_equals_greedy():
    B, gamma, V = 40, 6, 9000
    t = _ties(B, gamma + 1, V, "bf16", 13)
    a = torch.argmax(t[:, :gamma].float(), -1).to(torch.int32)
    x = torch.where(torch.rand((B, gamma), device=DEV) < 0.8, a, torch.zeros_like(a))
    parent = torch.tensor([-1] + list(range(gamma)), dtype=torch.int32, device=DEV)
    tok = torch.cat([torch.zeros((B, 1), dtype=torch.int32, device=DEV), x], 1)
    acc_t, out_t, _ = sv.spec_verify_tree_greedy(t, parent, tok, gamma)
    acc_g, out_g = sv.spec_verify_greedy(t, x)
    assert torch.equal(acc_t, acc_g) and torch.equal(out_t, out_g)


def test_tree_full_size():
    tr = W.make("tree_b64", device=DEV)
    acc, out, path = sv.spec_verify_tree_greedy(tr.target, tr.parent, tr.node_tokens, tr.max_depth)
    o_acc, o_out, o_path, flags = oracle_tree(tr.target, tr.parent, tr.node_tokens, tr.max_depth)
    assert _eq(acc, o_acc) and _eq(out, o_out) and _eq(path, o_path)
    assert (o_acc > 0).mean() > 0.3
    del tr
    torch.cuda.empty_cache()
