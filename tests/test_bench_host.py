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
