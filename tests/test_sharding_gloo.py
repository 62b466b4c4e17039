"""The N > 1 path on the CPU with two gloo ranks: the bench's process-group helpers
(barrier, max over ranks) and batch sharding by sequence ranges.  Sequences are
independent and their uniforms are keyed by the global sequence index, so the shards
concatenated equal the unsharded batch exactly -- no collective is needed on the data
path."""
import multiprocessing as mp
import socket

import numpy as np

import oracle
from speculative_decoding_verify_spec_gb300 import workloads as W

import dist_worker


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_shard_the_batch_exactly():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=dist_worker.run, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    t_max, acc, out = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert t_max == 11.0
    s = W.make_sample(10, 3, 700, dtype="bf16", seed=5, verify_seed=77, device="cpu")
    ref_acc, ref_out, _ = oracle.verify_sample(oracle.as_oracle_logits(s.target),
                                               oracle.as_oracle_logits(s.draft),
                                               s.draft_tokens.numpy(), s.temperature, s.seed)
    assert np.array_equal(np.array(acc), ref_acc)
    assert np.array_equal(np.array(out), ref_out)
