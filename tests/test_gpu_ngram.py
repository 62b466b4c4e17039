"""GPU parity of prompt-lookup (n-gram) drafting against the oracle, through the C ABI:
drafts and counts bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verify_spec_gb300 as sv
from speculative_decoding_verify_spec_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _check(h, L, n, k, pad):
    drafts, count = sv.spec_ngram_draft(h, L, n, k, pad)
    o_d, o_c = oracle.ngram_draft(h.cpu().numpy(), np.clip(L.cpu().numpy(), 0, h.shape[1]), n, k, pad)
    assert np.array_equal(count.cpu().numpy(), o_c)
    assert np.array_equal(drafts.cpu().numpy(), o_d)
    return count


@pytest.mark.parametrize("n,k,pad,alpha,T", [(1, 4, True, 3, 50), (1, 8, False, 50, 300), (2, 4, False, 3, 40),
                                             (3, 8, False, 4, 5000), (3, 0, True, 4, 100), (8, 16, True, 2, 9000),
                                             (64, 5, False, 2, 20000)])
def test_random_histories(n, k, pad, alpha, T):
    g = torch.Generator(device=DEV).manual_seed(n * 1000 + T)
    B = 200
    h = torch.randint(0, alpha, (B, T), generator=g, device=DEV, dtype=torch.int32)
    L = torch.randint(0, T + 1, (B,), generator=g, device=DEV, dtype=torch.int32)
    L[:6] = torch.tensor([0, 1, n, n + 1, T, T - 1], dtype=torch.int32)[:6].clamp(0, T)
    _check(h, L, n, k, pad)


def test_no_match_and_far_match():
    # a long history with distinct tokens has no earlier occurrence (a full scan); a single
    # occurrence at the very start is found across many chunks
    B, T = 8, 70000
    h = torch.arange(T, device=DEV, dtype=torch.int32).repeat(B, 1)
    L = torch.full((B,), T, device=DEV, dtype=torch.int32)
    for pad in (False, True):
        c = _check(h, L, 3, 6, pad)
        assert (c == (6 if pad else 0)).all()
    h[:, 0:3] = h[:, T - 3:T]
    c = _check(h, L, 3, 6, False)
    assert (c == 6).all()
    L[0] = T + 5  # clamped to the row
    L[1] = -2
    _check(h, L, 3, 6, True)


def test_workload():
    s = W.make("ngram_b256", device=DEV)
    c = _check(s.history, s.lengths, s.n, s.k, s.pad)
    assert (c > 0).float().mean() > 0.5
