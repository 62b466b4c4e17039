"""Host-side accounting of bench.py, on the CPU with stand-in calls: the accepted-length
histogram and the re-draw counts it reports beside the timings, and the roofline peak it
divides by."""
import json
import os

import torch

import bench


def test_acceptance_histogram_and_redraw_counts():
    B = 8
    acc = torch.zeros(B, dtype=torch.int32)
    steps_seen = []
    g = torch.Generator().manual_seed(3)

    def call():
        a = torch.randint(-1, 5, (B,), generator=g, dtype=torch.int32)
        acc.copy_(a)
        steps_seen.append(a.clone())

    states = iter([(2, 2, 0), (0, 0, 0), (5, 4, 4)])
    call.redraw_state = lambda: next(states)
    out = bench.acceptance_stats(call, acc, 3)
    seen = torch.cat(steps_seen)
    assert out["steps"] == 3 and out["sequences"] == 3 * B
    assert out["invalid"] == int((seen < 0).sum())
    hist = out["accepted_len_hist"]
    for v in range(5):
        assert (hist[v] if v < len(hist) else 0) == int((seen == v).sum())
    valid = seen[seen >= 0].double()
    assert abs(out["mean_accepted_len"] - float(valid.mean())) < 1e-12
    assert out["redraw_marked"] == 7 and out["redraw_redone"] == 6
    assert out["redraw_rate"] == 7 / (3 * B)
    assert out["redraw_status_nonzero"] == 1


def test_acceptance_without_redraw_hook():
    acc = torch.full((4,), 2, dtype=torch.int32)
    out = bench.acceptance_stats(lambda: None, acc, 2)
    assert out["accepted_len_hist"] == [0, 0, 8] and out["invalid"] == 0
    assert "redraw_marked" not in out


def test_hbm_peak_reads_measured_file():
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    peak, kind = bench.hbm_peak()
    if os.path.exists(path):
        with open(path) as f:
            assert peak == float(json.load(f)["hbm_gbs"]) and kind == "measured"
    else:
        assert (peak, kind) == (bench.FALLBACK_HBM_GBS, "fallback")


def test_oracle_legs_run_every_workload():
    """The CPU legs (cpu_baseline, --impl reference) call the oracle's rule for each
    workload: small versions of every one run, and report a histogram and flags where the
    rule has them."""
    from speculative_decoding_verify_spec_gb300 import workloads as W
    import __graft_entry__

    __graft_entry__._build_oracle()
    for name in W.WORKLOADS:
        mode = W.WORKLOADS[name]["mode"]
        ov = {"B": 3, "T": 600} if mode == "ngram" else {"B": 3, "V": 300}
        inputs = W.make(name, device="cpu", **ov)
        B, used, acc, flags = bench.oracle_run(name, inputs, 2)
        assert B == 3 and 1 <= used <= 2, name
        if mode == "ngram":
            assert acc is None and flags is None
            continue
        assert acc.shape == (3,) and (acc >= -1).all(), name
        out = bench.oracle_acceptance(acc, flags)
        assert sum(out["accepted_len_hist"]) + out["invalid"] == 3, name
        assert ("oracle_flags" in out) == (mode != "greedy"), name


def test_traffic_lines_are_keyed_to_their_kernels_sources():
    """A traffic capture is keyed to the files its kernel is built from: its translation unit,
    the headers it includes (transitively) and the host dispatch -- not the other kernels'
    sources; the single-sequence kernel shares the sampling unit's key."""
    names = lambda k: {os.path.basename(p) for p in bench.kernel_sources(k)}
    s = names("stats_tiles_kernel")
    assert {"sv_sample.cu", "sv_api.cu", "sv_refine.cuh", "sv_df.cuh", "sv_device.cuh", "spec_verify.h"} <= s
    assert not s & {"sv_tree_refine.cu", "sv_dfwalk.cuh", "sv_greedy.cu", "sv_level.cu"}
    assert names("max_tiles_kernel") >= {"sv_greedy.cu", "sv_api.cu"} and "sv_sample.cu" not in names("max_tiles_kernel")
    assert bench.source_digest("single_sample_kernel") == bench.source_digest("stats_tiles_kernel")
    assert bench.source_digest("level_kernel") != bench.source_digest("greedy_walk_kernel")
    # an unknown kernel is keyed to every source file
    assert "sv_tree_refine.cu" in names("tree_exp_kernel")
    # every committed line names a dominant kernel and parses
    for line in open(os.path.join(bench.ROOT, "profiles", "traffic.txt")):
        if line.strip() and not line.startswith("#"):
            k, w, dg, b = line.split()
            assert k in bench.KERNEL_SOURCE and len(dg) == 16 and int(b) > 0, line


def test_single_kernel_rule_matches_the_library_constants():
    """bench.py's copy of the dispatch rule for the one-kernel sampling call (its stage names
    and launch count) uses the library's tile sizes and tile limit: tiles of 32 lanes x 8
    vectors of 16 bytes, and kSingleTiles."""
    import re
    src = open(os.path.join(bench.ROOT, "speculative_decoding_verify_spec_gb300", "csrc", "sv_internal.h")).read()
    limit = int(re.search(r"constexpr int kSingleTiles = (\d+);", src).group(1))
    assert "inline int tile_elems_of(sv_dtype d) { return 32 * 8 * (16 / elem_bytes(d)); }" in src
    for dtype, tile in (("fp32", 1024), ("bf16", 2048)):
        for gamma in (0, 1, 4, 40):
            for V in (1, 1000, tile * 7 + 1, 128256):
                ntile = -(-V // tile)
                cfg = {"B": 1, "gamma": gamma, "V": V, "dtype": dtype}
                assert bench.single_kernel_call("sample", cfg) == ((2 * gamma + 1) * ntile <= limit)
                assert not bench.single_kernel_call("sample", dict(cfg, B=2))
                assert not bench.single_kernel_call("sample_lazy", cfg)


def test_source_digest_ignores_comments_and_blank_lines():
    """A comment or a blank line leaves a kernel's key unchanged; code does not."""
    a = "int f(int x) {  // twice\n    return 2 * x; /* doubled */\n}\n"
    b = "/* f */\nint f(int x) {\n\n    return 2 * x;\n}  // end\n"
    c = "int f(int x) {\n    return 3 * x;\n}\n"
    assert bench.strip_comments(a) == bench.strip_comments(b) != bench.strip_comments(c)
    assert bench.strip_comments('char *s = "a // b /* c */";') == 'char *s = "a // b /* c */";'
