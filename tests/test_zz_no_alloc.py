"""The greedy entry point that allocates nothing (spec_verify_greedy_noalloc).

It exists for callers that cannot give the library device memory while they run -- code
executing inside another runtime's step, where the host framework owns all buffers, or a
serving loop that must not call cudaMalloc after start-up.  Its results must equal those of
spec_verify_greedy (greedy verification is bit-exact), call after call, even though every
call reuses the same fixed device scratch.  This file is collected last on purpose.
"""
import pytest
import torch

import speculative_decoding_verify_spec_gb300 as sv
from speculative_decoding_verify_spec_gb300 import binding
from speculative_decoding_verify_spec_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    # two different problems back to back: the second call must not see the first's scratch
    cases = [(dict(B=96, gamma=6, V=50000, dtype="bf16", seed=21)),
             (dict(B=37, gamma=3, V=16385, dtype="fp32", seed=22))]
    for c in cases:
        g = W.make_greedy(c["B"], c["gamma"], c["V"], dtype=c["dtype"], seed=c["seed"], device=DEV)
        acc_ref, out_ref = sv.spec_verify_greedy(g.target, g.draft_tokens)
        acc, out = binding.spec_verify_greedy_noalloc(g.target, g.draft_tokens)
        torch.cuda.synchronize()
        assert torch.equal(acc, acc_ref)
        assert torch.equal(out, out_ref)


def test_full_size_greedy_fits_and_matches():
    g = W.make("greedy_b512", device=DEV)
    acc_ref, out_ref = sv.spec_verify_greedy(g.target, g.draft_tokens)
    acc, out = binding.spec_verify_greedy_noalloc(g.target, g.draft_tokens)
    torch.cuda.synchronize()
    assert torch.equal(acc, acc_ref) and torch.equal(out, out_ref)
    del g
    torch.cuda.empty_cache()


def test_problem_beyond_the_fixed_scratch_is_rejected_before_launch():
    # a broadcast view keeps the test small: 4096 sequences x 32 rows x 75 tiles of
    # partials need 75 MiB, more than the 4 MiB scratch
    row = torch.zeros((1, 1, 152064), dtype=torch.bfloat16, device=DEV)
    target = row.expand(4096, 32, 152064)
    tokens = torch.zeros((4096, 31), dtype=torch.int32, device=DEV)
    with pytest.raises(binding.SpecVerifyError, match="status 5"):
        binding.spec_verify_greedy_noalloc(target, tokens)
