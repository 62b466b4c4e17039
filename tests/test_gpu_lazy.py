"""GPU parity of the lazy entries (rows read only up to the stop point / at accepted
nodes) against the oracle and against the full entries, through the C ABI.

Bar: greedy and tree greedy bit-exact (lengths, tokens, paths); sampling equal to the
oracle wherever it raises no flag.  A bad row the walk never reads leaves the result as if
the row were good (the oracle and the full entries check every row, so those cases compare
against the same inputs with the row repaired).
"""
import numpy as np
import pytest
import torch

import speculative_decoding_verify_spec_gb300 as sv
from speculative_decoding_verify_spec_gb300 import binding
from speculative_decoding_verify_spec_gb300 import workloads as W

from parity_util import compare_sample, host, oracle_greedy, oracle_sample, oracle_tree, record_rates

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _greedy_case(B, gamma, V, dtype, seed, ties=False):
    g = torch.Generator(device=DEV).manual_seed(seed)
    if ties:  # small integers: many exact ties, lowest index must win
        t = torch.randint(-2, 3, (B, gamma + 1, V), generator=g, device=DEV).float()
    else:
        t = torch.randn((B, gamma + 1, V), generator=g, device=DEV) * 2
    t = t.to(torch.bfloat16 if dtype == "bf16" else torch.float32)
    a = torch.argmax(t.float(), dim=-1).to(torch.int32)
    x = torch.where(torch.rand((B, gamma), generator=g, device=DEV) < 0.8, a[:, :gamma],
                    torch.randint(0, V, (B, gamma), generator=g, device=DEV, dtype=torch.int32))
    return t.contiguous(), x.to(torch.int32).contiguous()


@pytest.mark.parametrize("B,gamma,V,dtype,ties", [(64, 0, 100, "fp32", False), (64, 1, 7, "bf16", True),
                                                   (200, 6, 2048, "bf16", True), (100, 6, 3001, "fp32", False),
                                                   (40, 12, 40000, "bf16", False)])
def test_greedy_lazy_matches(B, gamma, V, dtype, ties):
    t, x = _greedy_case(B, gamma, V, dtype, V + gamma, ties)
    acc, out = sv.spec_verify_greedy_lazy(t, x)
    f_acc, f_out = sv.spec_verify_greedy(t, x)
    o_acc, o_out = oracle_greedy(t, x)
    assert np.array_equal(acc.cpu().numpy(), o_acc) and np.array_equal(out.cpu().numpy(), o_out)
    assert torch.equal(acc, f_acc) and torch.equal(out, f_out)


def test_greedy_lazy_full_size_and_bad_rows():
    s = W.make("greedy_b512", device=DEV)
    acc, out = sv.spec_verify_greedy_lazy(s.target, s.draft_tokens)
    o_acc, o_out = oracle_greedy(s.target, s.draft_tokens)
    assert np.array_equal(acc.cpu().numpy(), o_acc) and np.array_equal(out.cpu().numpy(), o_out)
    # a NaN in a row the walk reads (row 0) invalidates; one past the stop row does not
    t, x = s.target[:8].clone(), s.draft_tokens[:8].clone()
    stop = acc[:8].cpu().numpy()
    t[0, 0, 5] = float("nan")
    later = [b for b in range(1, 8) if stop[b] < 6]
    for b in later:
        t[b, stop[b] + 1, 7] = float("nan")
    x[1, 0] = -3 if 1 not in later else x[1, 0]
    acc2, out2 = sv.spec_verify_greedy_lazy(t, x)
    a2 = acc2.cpu().numpy()
    assert a2[0] == -1 and (out2[0] == -1).all()
    for b in later:
        if b == 1 and x[1, 0] == -3:
            continue
        assert a2[b] == stop[b] and torch.equal(out2[b], out[b])


def test_tree_greedy_lazy_matches():
    s = W.make("tree_b64", device=DEV)
    acc, out, path = sv.spec_verify_tree_greedy_lazy(s.target, s.parent, s.node_tokens, s.max_depth)
    o = oracle_tree(s.target, s.parent, s.node_tokens, s.max_depth)
    assert np.array_equal(acc.cpu().numpy(), o[0]) and np.array_equal(out.cpu().numpy(), o[1])
    assert np.array_equal(path.cpu().numpy(), o[2])
    rs = np.random.RandomState(3)
    for N, V in ((1, 5), (12, 3), (40, 6), (64, 1000)):  # tiny V: duplicate matching siblings
        parent = [-1] + [int(rs.randint(0, v)) for v in range(1, N)]
        depth = [0] * N
        for v in range(1, N):
            depth[v] = depth[parent[v]] + 1
        B = 80
        g = torch.Generator(device=DEV).manual_seed(N * V)
        t = torch.randint(-2, 3, (B, N, V), generator=g, device=DEV).to(torch.bfloat16)
        a = torch.argmax(t.float(), dim=-1)
        tok = torch.randint(0, V, (B, N), generator=g, device=DEV, dtype=torch.int32)
        par = torch.tensor(parent, dtype=torch.int32, device=DEV)
        for v in range(1, N):
            m = torch.rand(B, generator=g, device=DEV) < 0.7
            tok[m, v] = a[m, parent[v]].to(torch.int32)
        D = max(depth)
        acc, out, path = sv.spec_verify_tree_greedy_lazy(t, par, tok, D)
        f = sv.spec_verify_tree_greedy(t, par, tok, D)
        o = oracle_tree(t, par, tok, D)
        for got, full, want in zip((acc, out, path), f, o[:3]):
            assert np.array_equal(got.cpu().numpy(), want) and torch.equal(got, full)


@pytest.mark.parametrize("name", ["sample_b1", "sample_b64", "sample_b256"])
def test_sample_lazy_matches_oracle(name):
    s = W.make(name, device=DEV)
    for off in range(3):
        acc, out = sv.spec_verify_sample_lazy(s.target, s.draft, s.draft_tokens, s.temperature, s.seed, off)
        o = oracle_sample(s.target, s.draft, s.draft_tokens, s.temperature, s.seed, off, diagnostics=True)
        compare_sample(acc, out, *o, label=f"lazy {name} offset {off}", record=True)
    del s
    torch.cuda.empty_cache()


def test_sample_lazy_small_and_edge_cases():
    for B, gamma, V, dtype, T in ((32, 0, 500, "fp32", 1.0), (64, 3, 4099, "bf16", 0.8), (48, 7, 777, "fp32", 1.3)):
        s = W.make_sample(B, gamma, V, dtype, recipe="normal", temperature=T, seed=V, verify_seed=5, device=DEV,
                          target_std=2.0, noise_std=1.0)
        acc, out = sv.spec_verify_sample_lazy(s.target, s.draft, s.draft_tokens, T, 5, 1)
        o = oracle_sample(s.target, s.draft, s.draft_tokens, T, 5, 1, diagnostics=True)
        compare_sample(acc, out, *o, label=f"lazy sample B={B} gamma={gamma} V={V} {dtype}", record=True)
    # identical rows: every draft accepted, bonus from row gamma
    s = W.make_sample(16, 4, 1000, "bf16", recipe="normal", temperature=1.0, seed=2, verify_seed=5, device=DEV,
                      target_std=2.0, noise_std=1.0)
    d = s.target[:, :4].contiguous()
    acc, out = sv.spec_verify_sample_lazy(s.target, d, s.draft_tokens, 1.0, 5)
    assert (acc == 4).all()


def test_sample_lazy_disagreements_are_below_one_in_ten_thousand():
    """40 rounds of the B=256 workload through the lazy entry: fewer than 0.01 % of the
    10,240 sequences disagree with the oracle; the double-float re-walk ran."""
    s = W.make("sample_b256", device=DEV)
    B, G1, V = s.target.shape
    ws = torch.empty(sv.spec_verify_workspace_size(binding.MODE_SAMPLE_LAZY, B, G1 - 1, V, binding.BF16),
                     dtype=torch.uint8, device=DEV)
    t, d, x = host(s.target), host(s.draft), s.draft_tokens.cpu().numpy()
    total = mism = flg = marked = 0
    flags = []
    for off in range(1, 41):
        acc, out = sv.spec_verify_sample_lazy(s.target, s.draft, s.draft_tokens, s.temperature, s.seed, off,
                                              workspace=ws)
        m, r, status, _ = binding.call_status(ws, binding.MODE_SAMPLE_LAZY, B, G1 - 1, V, binding.BF16)
        assert status == 0 and r == m
        marked += m
        o = oracle_sample(t, d, x, s.temperature, s.seed, off, diagnostics=True)
        n, mm, f, _ = compare_sample(acc, out, *o, label=f"lazy sample_b256 offset {off}")
        total, mism, flg = total + n, mism + mm, flg + f
        flags.append(o[2])
    record_rates("lazy sample_b256 x40 rounds", total, mism, flg, np.concatenate(flags), redraw_marked=marked)
    assert total == 10240
    assert marked > 0
    assert mism < 1e-4 * total, (mism, total)

