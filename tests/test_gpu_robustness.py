"""The library under serving conditions: its one software wait gives up with a status the
host can read (and the context stays usable), and every verify entry point can be captured
in a CUDA graph and replayed with the same results as an eager call."""
import time

import pytest
import torch

import speculative_decoding_verify_spec_gb300 as sv
from speculative_decoding_verify_spec_gb300 import binding
from speculative_decoding_verify_spec_gb300 import workloads as W

from parity_util import compare_sample, oracle_sample

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SV_ERR_TIMEOUT = 4


def test_bounded_wait_times_out_and_the_context_survives():
    t0 = time.perf_counter()
    assert binding.wait_selftest(2, 50_000) == SV_ERR_TIMEOUT  # nobody else arrives: 50 ms, then give up
    assert time.perf_counter() - t0 < 5.0
    assert binding.wait_selftest(1, 50_000) == 0                 # a barrier of one passes at once
    s = W.make_sample(16, 3, 2000, "bf16", recipe="normal", temperature=1.0, seed=3, verify_seed=5, device=DEV,
                      target_std=2.0, noise_std=1.0)
    acc, out = sv.spec_verify_sample(s.target, s.draft, s.draft_tokens, 1.0, 5, 1)
    o = oracle_sample(s.target, s.draft, s.draft_tokens, 1.0, 5, 1, diagnostics=True)
    compare_sample(acc, out, *o, label="after a timed-out wait")


def _graph_equals_eager(run, outs):
    """run(): one call writing into the preallocated tensors `outs`."""
    run()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    for o in outs:
        o.fill_(-7)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    for o in outs:
        o.fill_(-7)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for o in outs:
        o.fill_(-7)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, outs):
        assert torch.equal(a, b)


def test_entries_replay_from_a_cuda_graph():
    s = W.make_sample(64, 5, 32000, "bf16", recipe="normal", temperature=1.0, seed=7, verify_seed=5, device=DEV,
                      target_std=2.0, noise_std=1.0)
    B, G1, V = s.target.shape
    acc = torch.empty(B, dtype=torch.int32, device=DEV)
    out = torch.empty((B, G1), dtype=torch.int32, device=DEV)

    def ws(mode, rows):
        return torch.empty(sv.spec_verify_workspace_size(mode, B, rows, V, binding.BF16), dtype=torch.uint8,
                           device=DEV)

    w = ws(binding.MODE_SAMPLE, G1 - 1)
    _graph_equals_eager(lambda: sv.spec_verify_sample(s.target, s.draft, s.draft_tokens, 1.0, 5, 11, workspace=w,
                                                      accepted_len=acc, out_tokens=out), [acc, out])
    w = ws(binding.MODE_GREEDY, G1 - 1)
    _graph_equals_eager(lambda: sv.spec_verify_greedy(s.target, s.draft_tokens, workspace=w, accepted_len=acc,
                                                      out_tokens=out), [acc, out])
    w = ws(binding.MODE_SAMPLE_LAZY, G1 - 1)
    _graph_equals_eager(lambda: sv.spec_verify_sample_lazy(s.target, s.draft, s.draft_tokens, 1.0, 5, 12,
                                                           workspace=w, accepted_len=acc, out_tokens=out), [acc, out])
    w = ws(binding.MODE_TYPICAL, G1 - 1)
    _graph_equals_eager(lambda: sv.spec_verify_typical(s.target, s.draft_tokens, 1.0, 0.1, 0.3, 5, 13, workspace=w,
                                                       accepted_len=acc, out_tokens=out), [acc, out])
    w = ws(binding.MODE_SAMPLE_ONEHOT, G1 - 1)
    _graph_equals_eager(lambda: sv.spec_verify_sample_onehot(s.target, s.draft_tokens, 1.0, 5, 14, workspace=w,
                                                             accepted_len=acc, out_tokens=out), [acc, out])
    _graph_equals_eager(lambda: sv.spec_verify_greedy_lazy(s.target, s.draft_tokens, accepted_len=acc,
                                                           out_tokens=out), [acc, out])

    ts = W.make_tree_sample(16, 5000, "bf16", seed=8, device=DEV, N=64, without_replacement=True)
    Bt, N, Vt = ts.target.shape
    Wd = ts.max_depth + 1
    tacc = torch.empty(Bt, dtype=torch.int32, device=DEV)
    tout = torch.empty((Bt, Wd), dtype=torch.int32, device=DEV)
    tpath = torch.empty((Bt, Wd), dtype=torch.int32, device=DEV)
    w = torch.empty(sv.spec_verify_workspace_size(binding.MODE_TREE_SAMPLE, Bt, N, Vt, binding.BF16),
                    dtype=torch.uint8, device=DEV)
    _graph_equals_eager(lambda: sv.spec_verify_tree_sample(ts.target, ts.draft, ts.parent, ts.node_tokens,
                                                           ts.max_depth, 1.0, 9, 3, without_replacement=True,
                                                           workspace=w, accepted_len=tacc, out_tokens=tout,
                                                           out_path=tpath), [tacc, tout, tpath])
    w = torch.empty(sv.spec_verify_workspace_size(binding.MODE_TREE, Bt, N, Vt, binding.BF16),
                    dtype=torch.uint8, device=DEV)
    _graph_equals_eager(lambda: sv.spec_verify_tree_greedy(ts.target, ts.parent, ts.node_tokens, ts.max_depth,
                                                           workspace=w, accepted_len=tacc, out_tokens=tout,
                                                           out_path=tpath), [tacc, tout, tpath])
    _graph_equals_eager(lambda: sv.spec_verify_tree_greedy_lazy(ts.target, ts.parent, ts.node_tokens, ts.max_depth,
                                                                accepted_len=tacc, out_tokens=tout, out_path=tpath),
                        [tacc, tout, tpath])
