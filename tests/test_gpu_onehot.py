"""GPU parity of sampling verification against a one-hot draft distribution (the
prompt-lookup drafter's q) with the oracle, through the C ABI.

The oracle is the sampling oracle given draft rows that are -inf except 0 at each draft
(its q is then exactly one-hot).  Bar: lengths and tokens equal the oracle's on every
sequence it does not flag; over 10^4 sequences of the B=256 workload, disagreements of any
kind stay below 0.01 % (near-boundary final draws are redone in double-float).
"""
import numpy as np
import pytest
import torch

import speculative_decoding_verify_spec_gb300 as sv
from speculative_decoding_verify_spec_gb300 import binding
from speculative_decoding_verify_spec_gb300 import workloads as W

from parity_util import compare_sample, host, oracle_sample, record_rates

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def onehot_rows(x, V, like):
    """Draft logits [B, gamma, V]: -inf except 0 at each draft token (device tensor)."""
    B, g = x.shape
    d = torch.full((B, g, V), float("-inf"), device=DEV, dtype=like.dtype)
    if g:
        d.scatter_(2, x.long().unsqueeze(-1), 0.0)
    return d


def _case(B, gamma, V, dtype, seed, mask=0.0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    t = torch.randn((B, gamma + 1, V), generator=g, device=DEV) * 2
    if mask > 0:
        t.masked_fill_(torch.rand(t.shape, generator=g, device=DEV) < mask, float("-inf"))
        t[:, :, 0] = 0.0
    t = t.to(torch.bfloat16 if dtype == "bf16" else torch.float32).contiguous()
    q = torch.softmax(t.float() * 0.8 + torch.randn(t.shape, generator=g, device=DEV), -1)
    x = torch.multinomial(q[:, :gamma].reshape(-1, V), 1, generator=g).reshape(B, gamma).to(torch.int32) \
        if gamma > 0 else torch.zeros((B, 0), dtype=torch.int32, device=DEV)
    return t, x.contiguous()


@pytest.mark.parametrize("B,gamma,V,dtype,T,mask", [
    (64, 4, 1000, "fp32", 1.0, 0.0),
    (48, 6, 4099, "bf16", 0.7, 0.1),
    (40, 8, 32000, "bf16", 1.3, 0.0),
    (32, 0, 777, "fp32", 1.0, 0.0),
    (64, 5, 2048, "bf16", 1.0, 0.4),
])
def test_small_cases_match_oracle_and_full_entry(B, gamma, V, dtype, T, mask):
    t, x = _case(B, gamma, V, dtype, V + gamma, mask)
    d = onehot_rows(x, V, t)
    for off in range(3):
        acc, out = sv.spec_verify_sample_onehot(t, x, T, 13, off)
        o = oracle_sample(t, d, x, T, 13, off, diagnostics=True)
        compare_sample(acc, out, *o, label=f"one-hot q B={B} g={gamma} V={V} {dtype} T={T}", record=True)
        if gamma > 0:  # the full entry with the one-hot rows written out
            f_acc, f_out = sv.spec_verify_sample(t, d, x, T, 13, off)
            same = (f_acc == acc) & (f_out == out).all(1)
            flagged = torch.from_numpy(o[2] != 0).to(DEV)
            assert bool((same | flagged).all())


def test_bad_inputs_and_unread_rows():
    t, x = _case(6, 4, 500, "fp32", 5)
    x[:, 0] = 3
    t[:, 0, 3] = float("-inf")   # p(x_0) = 0: every sequence rejects at row 0
    t[0, 0, 7] = float("nan")    # a NaN in a row the rule reads
    t[1, 2, 1] = float("nan")    # ... and in one it never reads
    x[2, 3] = -1                 # a token out of range
    acc, out = sv.spec_verify_sample_onehot(t, x, 1.0, 4, 0)
    a = acc.cpu().numpy()
    assert a[0] == -1 and a[2] == -1 and (out[0] == -1).all() and (out[2] == -1).all()
    assert a[1] == 0 and (a[3:] == 0).all()
    assert (out[[1, 3, 4, 5], 0] != 3).all()  # the rejected draft is never the correction


def test_disagreements_are_below_one_in_ten_thousand():
    """40 rounds of the B=256 sampling workload's target rows and drafts, one-hot q."""
    s = W.make("sample_b256", device=DEV)
    B, G1, V = s.target.shape
    ws = torch.empty(sv.spec_verify_workspace_size(binding.MODE_SAMPLE_ONEHOT, B, G1 - 1, V, binding.BF16),
                     dtype=torch.uint8, device=DEV)
    t = host(s.target)
    d = host(onehot_rows(s.draft_tokens, V, s.target))
    xs = s.draft_tokens.cpu().numpy()
    total = mism = flg = marked = 0
    flags, lens = [], []
    for off in range(1, 41):
        acc, out = sv.spec_verify_sample_onehot(s.target, s.draft_tokens, s.temperature, s.seed, off, workspace=ws)
        m, r, status, _ = binding.call_status(ws, binding.MODE_SAMPLE_ONEHOT, B, G1 - 1, V, binding.BF16)
        assert status == 0 and r == m
        marked += m
        o = oracle_sample(t, d, xs, s.temperature, s.seed, off, diagnostics=True)
        n, mm, f, _ = compare_sample(acc, out, *o, label=f"one-hot sample_b256 offset {off}")
        total, mism, flg = total + n, mism + mm, flg + f
        flags.append(o[2])
        lens.append(acc.cpu().numpy())
    record_rates("one-hot q sample_b256 x40 rounds", total, mism, flg, np.concatenate(flags),
                 mean_accepted=float(np.concatenate(lens).mean()), redraw_marked=marked)
    assert total == 10240
    assert marked > 0
    assert mism < 1e-4 * total, (mism, total)
