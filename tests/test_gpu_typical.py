"""GPU parity of typical acceptance (Medusa's relaxed rule) against the oracle, through the
C ABI.

Bar: accepted_len and every token equal the oracle's, except on sequences the oracle flags
(a target probability within 1e-5 of its threshold, or a draw within 1e-5 of a CDF
boundary); over 10^4 sequences of the B=256 workload, disagreements of any kind stay below
0.01 % (near-boundary final draws are redone in double-float).  The rule's form and constants are a reading of the pages (parity of the constants
unpinned); the oracle's pins fix the rest.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_verify_spec_gb300 as sv
from speculative_decoding_verify_spec_gb300 import binding
from speculative_decoding_verify_spec_gb300 import workloads as W

import oracle
from parity_util import compare_sample, host, record_rates

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _oracle(target, tokens, T, eps, delta, seed, offset):
    """The oracle on the same inputs, with the parameters as the C ABI receives them (fp32)."""
    f = lambda v: float(np.float32(v))  # noqa: E731
    acc, out, flags, _ = oracle.default().verify_typical(host(target), tokens.cpu().numpy(), f(T), f(eps), f(delta),
                                                         seed, offset)
    return acc, out, flags


def _case(B, gamma, V, dtype, seed, std=2.0, mask=0.0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    t = torch.randn((B, gamma + 1, V), generator=g, device=DEV) * std
    if mask > 0:
        m = torch.rand(t.shape, generator=g, device=DEV) < mask
        t.masked_fill_(m, float("-inf"))
        t[:, :, 0] = 0.0
    t = t.to(torch.bfloat16 if dtype == "bf16" else torch.float32).contiguous()
    p = torch.softmax(t.float(), -1)
    x = torch.multinomial(p[:, :gamma].reshape(-1, V), 1, generator=g).reshape(B, gamma).to(torch.int32) \
        if gamma > 0 else torch.zeros((B, 0), dtype=torch.int32, device=DEV)
    return t, x.contiguous()


@pytest.mark.parametrize("B,gamma,V,dtype,T,eps,delta,mask", [
    (64, 4, 1000, "fp32", 1.0, 0.09, 0.3, 0.0),
    (48, 6, 4099, "bf16", 0.7, 0.05, 0.5, 0.1),
    (40, 8, 32000, "bf16", 1.3, 0.2, 0.2, 0.0),
    (32, 0, 777, "fp32", 1.0, 0.1, 0.3, 0.0),
    (64, 5, 2048, "bf16", 1.0, 0.0, 0.3, 0.3),   # epsilon = 0: every finite-logit draft accepted
    (64, 5, 3001, "fp32", 1.0, 2.0, 1e30, 0.0),  # threshold 2 > any p: the first token from p_0
])
def test_small_cases_match_oracle(B, gamma, V, dtype, T, eps, delta, mask):
    t, x = _case(B, gamma, V, dtype, V + gamma, mask=mask)
    for off in range(3):
        acc, out = sv.spec_verify_typical(t, x, T, eps, delta, 11, off)
        o = _oracle(t, x, T, eps, delta, 11, off)
        compare_sample(acc, out, *o, label=f"typical B={B} g={gamma} V={V} {dtype} eps={eps} delta={delta}",
                       record=True)
    if eps == 0.0:
        dead = (t.float().gather(2, torch.cat([x, x[:, :1]], 1).long().unsqueeze(-1))[:, :gamma, 0] == float("-inf"))
        want = torch.where(dead.any(1), dead.int().argmax(1), torch.full_like(dead[:, 0], gamma, dtype=torch.int64))
        assert torch.equal(acc.long(), want)
    if eps == 2.0:
        assert (acc == 0).all()


def test_bad_inputs_and_unread_rows():
    t, x = _case(6, 4, 500, "fp32", 5, mask=0.0)
    x[:, 0] = 0
    t[:, 0, 0] = float("-inf")     # the first draft is ruled out: every sequence stops at row 0
    t[0, 0, 7] = float("nan")      # a NaN in a row the rule reads
    t[1, 2, 3] = float("nan")      # ... and in one it never reads
    x[2, 3] = 500                  # a token out of range
    acc, out = sv.spec_verify_typical(t, x, 1.0, 0.0, 0.3, 4, 0)
    o = _oracle(t, x, 1.0, 0.0, 0.3, 4, 0)
    compare_sample(acc, out, *o, label="typical bad inputs", record=True)
    a = acc.cpu().numpy()
    assert a[0] == -1 and a[2] == -1 and a[1] == 0 and (a[3:] == 0).all()


def test_unaligned_rows():
    base, x = _case(16, 5, 3001, "bf16", 21)
    B, G1, V = base.shape
    big = torch.zeros((B, G1, V + 3), device=DEV, dtype=torch.bfloat16)
    big[:, :, 1:V + 1] = base
    t = big[:, :, 1:V + 1]
    acc, out = sv.spec_verify_typical(t, x, 0.8, 0.1, 0.3, 21, 2)
    o = _oracle(base, x, 0.8, 0.1, 0.3, 21, 2)
    compare_sample(acc, out, *o, label="typical unaligned rows", record=True)


def test_disagreements_are_below_one_in_ten_thousand():
    """40 rounds of the B=256 workload (fresh uniforms per round via the offset)."""
    s = W.make("typical_b256", device=DEV)
    cfg = W.WORKLOADS["typical_b256"]
    B, G1, V = s.target.shape
    ws = torch.empty(sv.spec_verify_workspace_size(binding.MODE_TYPICAL, B, G1 - 1, V, binding.BF16),
                     dtype=torch.uint8, device=DEV)
    t, xs = host(s.target), s.draft_tokens.cpu().numpy()
    orc = oracle.default()
    total = mism = flg = marked = 0
    flags, lens = [], []
    for off in range(1, 41):
        acc, out = sv.spec_verify_typical(s.target, s.draft_tokens, s.temperature, cfg["epsilon"], cfg["delta"],
                                          s.seed, off, workspace=ws)
        m, r, status, _ = binding.call_status(ws, binding.MODE_TYPICAL, B, G1 - 1, V, binding.BF16)
        assert status == 0 and r == m
        marked += m
        o = orc.verify_typical(t, xs, float(np.float32(s.temperature)), float(np.float32(cfg["epsilon"])),
                               float(np.float32(cfg["delta"])), s.seed, off)
        n, m, f, _ = compare_sample(acc, out, *o[:3], label=f"typical_b256 offset {off}")
        total, mism, flg = total + n, mism + m, flg + f
        flags.append(o[2])
        lens.append(acc.cpu().numpy())
    record_rates("typical_b256 x40 rounds", total, mism, flg, np.concatenate(flags),
                 mean_accepted=float(np.concatenate(lens).mean()), redraw_marked=marked)
    assert total == 10240
    assert marked > 0  # the re-draw is exercised
    assert mism < 1e-4 * total, (mism, total)
