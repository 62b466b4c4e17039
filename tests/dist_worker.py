"""Worker for the world_size-2 gloo test (spawned; CPU only)."""
import os


def run(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    import oracle
    from speculative_decoding_verify_spec_gb300 import workloads as W

    r, w, _ = bench.dist_setup("gloo")
    assert (r, w) == (rank, world)
    # the bench's max-over-ranks timing reduction
    t_max = bench.max_over_ranks(10.0 + rank, w, "cpu")
    bench.barrier(w)
    # shard a batch by contiguous sequence ranges; the global index b0 keys the uniforms
    s = W.make_sample(10, 3, 700, dtype="bf16", seed=5, verify_seed=77, device="cpu")
    B = s.target.shape[0]
    lo, hi = rank * B // world, (rank + 1) * B // world
    t = oracle.as_oracle_logits(s.target)[lo:hi]
    d = oracle.as_oracle_logits(s.draft)[lo:hi]
    x = s.draft_tokens.numpy()[lo:hi]
    acc, out, _ = oracle.verify_sample(t, d, x, s.temperature, s.seed, 0, b0=lo)
    g = [None] * w
    dist.all_gather_object(g, (lo, acc.tolist(), out.tolist()))
    dist.barrier()
    dist.destroy_process_group()
    if rank == 0:
        g.sort()
        out_q.put((t_max, sum((p[1] for p in g), []), sum((p[2] for p in g), [])))
