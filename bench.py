#!/usr/bin/env python
"""Throughput of the speculative-decoding verification step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one verify call over one batch of the workload (default: sampling verify,
B=256, V=128256, gamma=8, bf16 logits, T=0.7 -- every kernel of the sampling path).  The
greedy (B=512, V=152064, gamma=6) and tree (B=64, N=64, V=128256) workloads are measured
the same way and reported under "modes".  Inputs are synthetic and resident in HBM; each
step reads more than L2 holds, so no flush is needed between steps.

Under torchrun (N > 1) each rank verifies its own batch (sequences are independent: weak
scaling, no collective on the data path); the time is the max over ranks.

--impl reference times the oracle (plain fp64 C, tests' reference) on the host cores over
a bounded sample of the same workload, rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "sample_b256"
# the five configurations the metric is quoted on (C1 .. C5), then the NEXT rules
CONFIGS = {"sample_b1": "C1", "sample_b64": "C2", "sample_b256": "C3", "greedy_b512": "C4", "tree_b64": "C5"}
SECONDARY = ["sample_b1", "sample_b64", "greedy_b512", "tree_b64", "tree_sample_b64", "sample_b256_lazy",
             "typical_b256", "onehot_b256", "greedy_b512_lazy", "tree_b64_lazy", "ngram_b256"]
METRIC = "verified seqs/s"
UNIT = "seqs/s"
FALLBACK_HBM_GBS = 6800.0
DOMINANT_KERNEL = {"sample": "stats_tiles_kernel", "greedy": "max_tiles_kernel",
                   "tree": "max_tiles_kernel", "tree_sample": "tree_sample_kernel",
                   "sample_lazy": "level_kernel", "greedy_lazy": "greedy_walk_kernel",
                   "tree_lazy": "greedy_walk_kernel", "ngram": "ngram_draft_kernel",
                   "typical": "level_kernel", "onehot": "level_kernel"}
# A sampling call with B = 1 whose 2 gamma + 1 rows have at most 256 tiles of 4 KB runs as
# one kernel (single_sample_kernel); its stage events 2..4 are recorded right after it.
SINGLE_STAGES = ["one_kernel", "none_1", "none_2", "none_3"]


def single_kernel_call(mode: str, cfg: dict) -> bool:
    tile = 1024 if cfg["dtype"] == "fp32" else 2048
    return mode == "sample" and cfg["B"] == 1 and (2 * cfg["gamma"] + 1) * -(-cfg["V"] // tile) <= 256
STAGE_STEPS = 200  # steps timed kernel by kernel (after the headline steps)
ACCEPT_STEPS = 16  # untimed steps whose accepted lengths and re-draw counts are read back
STAGES = {"sample": ["row_stats", "decide", "residual_mass", "draw_redraw"],
          "greedy": ["argmax", "finalize"], "tree": ["argmax", "finalize"], "tree_sample": ["walk", "rewalk_exp", "rewalk"],
          "sample_lazy": ["walk", "residual_mass", "draw_redraw"], "greedy_lazy": ["walk"], "tree_lazy": ["walk"],
          "ngram": ["draft"], "typical": ["walk", "draw_redraw"], "onehot": ["walk", "draw_redraw"]}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--no-modes", action="store_true", help="skip the greedy / tree workloads")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=30)
    p.add_argument("--batch", type=int, default=None,
                   help="override the workload's batch size (small profiling cases)")
    return p.parse_args()


# ----------------------------------------------------------------------------------------
# process group
# ----------------------------------------------------------------------------------------
def dist_setup(backend="nccl"):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            out_dir = os.environ.get("SV_BENCH_OUT")  # where to keep the raw samples, if anywhere
            if out_dir:
                os.makedirs(out_dir, exist_ok=True)
                self.path = os.path.join(out_dir, f"clocks_gpu{self.gpu}.csv")
                self.f = open(self.path, "w")
            else:
                self.f = tempfile.NamedTemporaryFile("w", suffix=".csv", delete=False)
                self.path = self.f.name
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:  # no nvidia-smi: no clock record
            self.proc = None
            if self.path and not os.environ.get("SV_BENCH_OUT"):
                self.f.close()
                os.unlink(self.path)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            lines = f.readlines()
        if not os.environ.get("SV_BENCH_OUT"):
            os.unlink(self.path)
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1].split()[0]))
                mx = float(parts[2].split()[0])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------------------
# measured peaks and committed ncu traffic
# ----------------------------------------------------------------------------------------
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# the translation unit that defines each dominant kernel
KERNEL_SOURCE = {"stats_tiles_kernel": "sv_sample.cu", "single_sample_kernel": "sv_sample.cu",
                 "max_tiles_kernel": "sv_greedy.cu", "level_kernel": "sv_level.cu",
                 "greedy_walk_kernel": "sv_lazy.cu"}


def kernel_sources(kernel: str) -> list:
    """The files a kernel's code and launch come from: its translation unit, every header it
    includes (transitively, from csrc/ and include/), and the host dispatch sv_api.cu with its
    includes.  Every source file for a kernel not in KERNEL_SOURCE."""
    csrc = os.path.join(ROOT, "speculative_decoding_verify_spec_gb300", "csrc")
    inc = os.path.join(ROOT, "include")
    if kernel not in KERNEL_SOURCE:
        return sorted(os.path.join(csrc, n) for n in os.listdir(csrc) if n.endswith((".cu", ".cuh", ".h")))
    seen, todo = set(), [os.path.join(csrc, KERNEL_SOURCE[kernel]), os.path.join(csrc, "sv_api.cu")]
    while todo:
        path = todo.pop()
        if path in seen or not os.path.exists(path):
            continue
        seen.add(path)
        for line in open(path, encoding="utf-8"):
            line = line.strip()
            if line.startswith("#include \""):
                name = line.split('"')[1]
                todo += [os.path.join(csrc, name), os.path.join(inc, name)]
    return sorted(seen)


def strip_comments(text: str) -> str:
    """C/C++ source without its comments and blank lines, each line stripped (string and
    character literals kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # a literal, to its closing quote
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.strip() for line in "".join(out).splitlines() if line.strip())


def source_digest(kernel: str = "") -> str:
    """A 16-hex-digit SHA-256 prefix over the code of the kernel's sources (kernel_sources,
    comments left out): a traffic capture stays valid while that code is unchanged."""
    h = hashlib.sha256()
    for path in kernel_sources(kernel):
        with open(path, encoding="utf-8") as f:
            h.update(os.path.basename(path).encode() + b"\0" + strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from profiles/traffic.txt, if the
    capture was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    digest = source_digest(kernel)
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and \
                parts[1] == workload and parts[2] == digest:
            return float(parts[3])
    return None


# ----------------------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------------------
def kernel_bytes(name: str, **ov) -> int:
    """Algorithmic bytes of the dominant kernel per launch: every logit it streams, once."""
    from speculative_decoding_verify_spec_gb300 import workloads as W
    cfg = W.WORKLOADS[name]
    if cfg["mode"] == "ngram":
        return W.logical_bytes(name, **ov)
    s = 2 if cfg["dtype"] == "bf16" else 4
    return W.rows(name, **ov) * cfg["V"] * s


def make_call(name, inputs, dev, **ov):
    """A closure that runs one verify call of the workload into preallocated outputs."""
    import torch
    import speculative_decoding_verify_spec_gb300 as sv
    from speculative_decoding_verify_spec_gb300 import binding
    from speculative_decoding_verify_spec_gb300 import workloads as W

    cfg = dict(W.WORKLOADS[name])
    cfg.update(ov)
    mode = cfg["mode"]
    B, V = cfg["B"], cfg["V"]
    lazy = cfg.get("lazy", False)
    if mode == "ngram":
        drafts = torch.empty((B, cfg["k"]), dtype=torch.int32, device=dev)
        count = torch.empty(B, dtype=torch.int32, device=dev)

        def call(history=inputs.history, lengths=inputs.lengths):
            return sv.spec_ngram_draft(history, lengths, inputs.n, inputs.k, inputs.pad, drafts=drafts, count=count)
        return call, (count, drafts)
    dt = binding.BF16 if cfg["dtype"] == "bf16" else binding.FP32
    if mode == "sample" and cfg.get("typical"):
        g = cfg["gamma"]
        ws = torch.empty(sv.spec_verify_workspace_size(binding.MODE_TYPICAL, B, g, V, dt),
                         dtype=torch.uint8, device=dev)
        acc = torch.empty(B, dtype=torch.int32, device=dev)
        out = torch.empty((B, g + 1), dtype=torch.int32, device=dev)
        step_counter = [0]

        def call(target=inputs.target, tokens=inputs.draft_tokens):
            step_counter[0] += 1
            return sv.spec_verify_typical(target, tokens, inputs.temperature, cfg["epsilon"], cfg["delta"],
                                          inputs.seed, step_counter[0], workspace=ws, accepted_len=acc,
                                          out_tokens=out)
        call.redraw_state = lambda: binding.call_status(ws, binding.MODE_TYPICAL, B, g, V, dt)[:3]
        return call, (acc, out)
    if mode == "sample" and cfg.get("onehot"):
        g = cfg["gamma"]
        ws = torch.empty(sv.spec_verify_workspace_size(binding.MODE_SAMPLE_ONEHOT, B, g, V, dt),
                         dtype=torch.uint8, device=dev)
        acc = torch.empty(B, dtype=torch.int32, device=dev)
        out = torch.empty((B, g + 1), dtype=torch.int32, device=dev)
        step_counter = [0]

        def call(target=inputs.target, tokens=inputs.draft_tokens):
            step_counter[0] += 1
            return sv.spec_verify_sample_onehot(target, tokens, inputs.temperature, inputs.seed, step_counter[0],
                                                workspace=ws, accepted_len=acc, out_tokens=out)
        call.redraw_state = lambda: binding.call_status(ws, binding.MODE_SAMPLE_ONEHOT, B, g, V, dt)[:3]
        return call, (acc, out)
    if mode == "sample" and lazy:
        g = cfg["gamma"]
        ws = torch.empty(sv.spec_verify_workspace_size(binding.MODE_SAMPLE_LAZY, B, g, V, dt),
                         dtype=torch.uint8, device=dev)
        acc = torch.empty(B, dtype=torch.int32, device=dev)
        out = torch.empty((B, g + 1), dtype=torch.int32, device=dev)
        step_counter = [0]

        def call(target=inputs.target, draft=inputs.draft, tokens=inputs.draft_tokens):
            step_counter[0] += 1
            return sv.spec_verify_sample_lazy(target, draft, tokens, inputs.temperature, inputs.seed,
                                              step_counter[0], workspace=ws, accepted_len=acc,
                                              out_tokens=out)
        call.redraw_state = lambda: binding.call_status(ws, binding.MODE_SAMPLE_LAZY, B, g, V, dt)[:3]
        return call, (acc, out)
    if mode == "greedy" and lazy:
        g = cfg["gamma"]
        acc = torch.empty(B, dtype=torch.int32, device=dev)
        out = torch.empty((B, g + 1), dtype=torch.int32, device=dev)

        def call(target=inputs.target, tokens=inputs.draft_tokens):
            return sv.spec_verify_greedy_lazy(target, tokens, accepted_len=acc, out_tokens=out)
        return call, (acc, out)
    if mode == "tree" and lazy:
        acc = torch.empty(B, dtype=torch.int32, device=dev)
        out = torch.empty((B, inputs.max_depth + 1), dtype=torch.int32, device=dev)
        path = torch.empty((B, inputs.max_depth + 1), dtype=torch.int32, device=dev)

        def call(target=inputs.target, tokens=inputs.node_tokens):
            return sv.spec_verify_tree_greedy_lazy(target, inputs.parent, tokens, inputs.max_depth,
                                                   accepted_len=acc, out_tokens=out, out_path=path)
        return call, (acc, out, path)
    if mode == "sample":
        g = cfg["gamma"]
        ws = torch.empty(sv.spec_verify_workspace_size(binding.MODE_SAMPLE, B, g, V, dt),
                         dtype=torch.uint8, device=dev)
        acc = torch.empty(B, dtype=torch.int32, device=dev)
        out = torch.empty((B, g + 1), dtype=torch.int32, device=dev)
        step_counter = [0]

        def call(target=inputs.target, draft=inputs.draft, tokens=inputs.draft_tokens):
            step_counter[0] += 1
            return sv.spec_verify_sample(target, draft, tokens, inputs.temperature, inputs.seed,
                                         step_counter[0], workspace=ws, accepted_len=acc,
                                         out_tokens=out)

        call.redraw_state = lambda: binding.call_status(ws, binding.MODE_SAMPLE, B, g, V, dt)[:3]
        return call, (acc, out)
    if mode == "greedy":
        g = cfg["gamma"]
        ws = torch.empty(sv.spec_verify_workspace_size(binding.MODE_GREEDY, B, g, V, dt),
                         dtype=torch.uint8, device=dev)
        acc = torch.empty(B, dtype=torch.int32, device=dev)
        out = torch.empty((B, g + 1), dtype=torch.int32, device=dev)

        def call(target=inputs.target, tokens=inputs.draft_tokens):
            return sv.spec_verify_greedy(target, tokens, workspace=ws, accepted_len=acc, out_tokens=out)
        return call, (acc, out)
    N = cfg["N"]
    if mode == "tree_sample":
        ws = torch.empty(sv.spec_verify_workspace_size(binding.MODE_TREE_SAMPLE, B, N, V, dt),
                         dtype=torch.uint8, device=dev)
        acc = torch.empty(B, dtype=torch.int32, device=dev)
        out = torch.empty((B, inputs.max_depth + 1), dtype=torch.int32, device=dev)
        path = torch.empty((B, inputs.max_depth + 1), dtype=torch.int32, device=dev)
        step_counter = [0]

        def call(target=inputs.target, tokens=inputs.node_tokens, draft=inputs.draft):
            step_counter[0] += 1
            return sv.spec_verify_tree_sample(target, draft, inputs.parent, tokens,
                                              inputs.max_depth, inputs.temperature, inputs.seed,
                                              step_counter[0],
                                              without_replacement=inputs.without_replacement,
                                              workspace=ws, accepted_len=acc, out_tokens=out,
                                              out_path=path)
        call.redraw_state = lambda: binding.call_status(ws, binding.MODE_TREE_SAMPLE, B, N, V, dt)[:3]
        return call, (acc, out, path)
    ws = torch.empty(sv.spec_verify_workspace_size(binding.MODE_TREE, B, N, V, dt),
                     dtype=torch.uint8, device=dev)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    out = torch.empty((B, inputs.max_depth + 1), dtype=torch.int32, device=dev)
    path = torch.empty((B, inputs.max_depth + 1), dtype=torch.int32, device=dev)

    def call(target=inputs.target, tokens=inputs.node_tokens):
        return sv.spec_verify_tree_greedy(target, inputs.parent, tokens, inputs.max_depth,
                                          workspace=ws, accepted_len=acc, out_tokens=out,
                                          out_path=path)
    return call, (acc, out, path)


def acceptance_stats(call, acc, steps):
    """Untimed: the accepted-length histogram over `steps` further calls (each with its own
    offset where the rule samples), and for the sampling rules how many sequences the
    extended-precision pass had to re-do -- the GPU's counterpart of the oracle's
    tolerance flags."""
    import torch
    seen = []
    marked = redone = 0
    status = []
    for _ in range(steps):
        call()
        seen.append(acc.long().clone())
        if hasattr(call, "redraw_state"):
            m, r, st = call.redraw_state()
            marked += m
            redone += r
            status.append(st)
    seqs = steps * acc.numel()
    hist = torch.bincount(torch.cat(seen) + 1).cpu()  # bin 0 counts invalid sequences (-1)
    out = {"steps": steps, "sequences": seqs, "invalid": int(hist[0]),
           "accepted_len_hist": [int(x) for x in hist[1:]],
           "mean_accepted_len": float((hist[1:] * torch.arange(len(hist) - 1)).sum()) / max(1, seqs - int(hist[0]))}
    if hasattr(call, "redraw_state"):
        out.update({"redraw_marked": marked, "redraw_redone": redone, "redraw_rate": marked / seqs,
                    "redraw_status_nonzero": sum(1 for x in status if x != 0)})
    return out


def step_distribution(call, n=200):
    """Per-step times (ms) of n calls, each bracketed by its own events: p10 / p50 / p90."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in evs:
        a.record()
        call()
        b.record()
    torch.cuda.synchronize()
    t = sorted(a.elapsed_time(b) for a, b in evs)
    return {"p10_ms": t[n // 10], "p50_ms": t[n // 2], "p90_ms": t[(9 * n) // 10], "steps": n}


def graph_time(call, per_graph=20, replays=50):
    """The same calls captured in one CUDA graph (per_graph calls, each with its own
    offset) and replayed: ms per call."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            call()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(per_graph):
            call()
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(replays):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / (replays * per_graph)


def l2_bytes(dev) -> int:
    import torch
    return int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (129 << 20))


def measure(name, steps, warmup, rank, world, dev, peak, peak_kind, batch=None, detail=False, graph=False):
    import torch
    from speculative_decoding_verify_spec_gb300 import binding
    from speculative_decoding_verify_spec_gb300 import workloads as W

    cfg = dict(W.WORKLOADS[name])
    ov = {} if batch is None else {"B": batch}
    cfg.update(ov)
    mode = cfg["mode"]
    inputs = W.make(name, device=dev, input_seed=cfg["input_seed"] + 7919 * rank, **ov)
    call, outs = make_call(name, inputs, dev, **ov)
    logical = W.logical_bytes(name, **ov)
    # Cold L2: a batch that fits in L2 (but is not just a few KB of launch latency) is timed
    # over rotating copies of its inputs totalling at least 4x L2, so every step reads from
    # HBM as a larger batch would.
    rotate, l2_note = 1, f"inputs larger than L2 ({logical / 1e9:.2f} GB read per step), no flush"
    L2 = l2_bytes(dev)
    if logical <= L2 and mode == "sample" and logical >= (1 << 20):
        rotate = -(-4 * L2 // logical)
        l2_note = (f"cold L2: {rotate} rotating copies of the inputs ({rotate * logical / 1e6:.0f} MB, "
                   f">= 4x the {L2 >> 20} MB L2), one per step")
    elif logical < (1 << 20):
        l2_note = f"L2-resident ({logical} B per step): launch-latency bound, no flush"
    copies = [inputs] + [W.make(name, device=dev, input_seed=cfg["input_seed"] + 7919 * rank, **ov)
                         for _ in range(rotate - 1)]

    def timed_call(k):
        if rotate == 1:
            return call()
        c = copies[k % rotate]
        return call(c.target, c.draft, c.draft_tokens)
    if cfg.get("lazy"):
        mode = mode + "_lazy"
    if cfg.get("typical"):
        mode = "typical"
    if cfg.get("onehot"):
        mode = "onehot"
    nst = len(STAGES[mode])
    if mode == "sample" and cfg["gamma"] == 0:
        nst = 5
    for _ in range(max(3, warmup)):
        call()
    torch.cuda.synchronize()
    # the timed steps: nothing but the calls (events between a call's kernels would keep
    # each kernel from being scheduled while the previous one drains)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record()
    for k in range(steps):
        timed_call(k)
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    ms = start.elapsed_time(end)
    ms_max = max_over_ranks(ms, world, dev)
    # then the per-kernel breakdown on separate steps, with the library's stage events
    # recorded on the call's stream around every kernel
    ksteps = min(steps, STAGE_STEPS)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(ksteps)]
    for row in ev:
        for e in row:
            e.record()
    torch.cuda.synchronize()
    for k in range(ksteps):
        binding.set_stage_events(ev[k])
        timed_call(k)
    binding.set_stage_events(None)
    torch.cuda.synchronize()
    stage_ms = [sum(ev[k][s].elapsed_time(ev[k][s + 1]) for k in range(ksteps)) / ksteps
                for s in range(nst)]
    extra = {}
    if mode != "ngram":
        try:  # reported beside the timings, never in place of them
            extra["acceptance"] = acceptance_stats(call, outs[0], ACCEPT_STEPS)
        except Exception as exc:
            extra["acceptance"] = {"error": f"{type(exc).__name__}: {exc}"[:200]}
    if detail:  # the per-step spread
        extra["step_spread"] = step_distribution(call)
    if detail or graph:  # the same step replayed from a CUDA graph
        try:
            gms = graph_time(call)
            extra["graph"] = {"ms_per_step": gms, "value": world * cfg["B"] / (gms / 1e3),
                              "note": "20 calls (20 offsets) captured in one graph, replayed 50 times"}
        except Exception as exc:  # capture is reported, not required
            extra["graph"] = {"error": f"{type(exc).__name__}: {exc}"[:200]}
    ms_step = ms_max / steps
    B = cfg["B"]
    value = world * B / (ms_step / 1e3)
    kb = kernel_bytes(name, **ov)
    dom_ms = stage_ms[0]
    achieved = kb / (dom_ms / 1e3) / 1e9
    single = single_kernel_call(mode, cfg)
    kernel = "single_sample_kernel" if single else DOMINANT_KERNEL[mode]
    stage_names = SINGLE_STAGES if single else STAGES[mode]
    acc = outs[0].float()
    res = {
        "workload": W.DESCRIPTIONS[name], "value": value, "unit": UNIT, "ms_per_step": ms_step,
        "steps": steps, "rows_per_s": world * W.rows(name, **ov) / (ms_step / 1e3),
        "hbm_gbs_step": logical / (ms_step / 1e3) / 1e9,
        "frac_of_8tbs_step": logical / (ms_step / 1e3) / 8e12,
        "stages_ms": dict(zip(stage_names, stage_ms)), "l2": l2_note,
        "mean_accepted_len": float(acc[acc >= 0].mean().item()) if (acc >= 0).any() else None,
        "roofline": {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind + " copy (read+write) bandwidth", "unit": "GB/s",
                     "frac": achieved / peak,
                     "bytes_per_launch": kb,
                     "traffic": committed_traffic(kernel, name)},
        "gpu_launches": steps * (1 if single else nst if mode != "sample" or cfg["gamma"] > 0 else 4),
        **extra,
    }
    if mode == "tree_sample":
        # the walk reads only the rows of the nodes it reaches: the every-row byte count of
        # the metric does not apply, and the kernel is bound by exponentials and latency
        res.update({"hbm_gbs_step": None, "frac_of_8tbs_step": None, "roofline": None,
                    "lazy": "a cluster of CTAs per sequence reads only the rows of the nodes its walk reaches",
                    "mean_path_nodes": float(acc[acc >= 0].mean().item() + 1) if (acc >= 0).any() else None})
    if mode == "ngram":
        res.update({"rows_per_s": None, "roofline": None, "mean_accepted_len": None,
                    "mean_drafts": float(outs[0].float().mean().item()),
                    "bytes_note": "every history token once; the search stops at the first chunk holding a match"})
    if mode.endswith("_lazy") or mode in ("typical", "onehot"):
        # bytes the walk kernel needs to read in the last step, from its outputs: chain greedy
        # reads rows 0..k, tree greedy the rows of the accepted nodes (at least the path), the
        # level walks target rows 0..k (and for the sampling chain draft rows
        # 0..min(k, gamma-1)); the sampling chain's step then reads 2 rows for the residual
        # (k < gamma) or 1 for the bonus, the other level walks row k once more for the draw
        s = 2 if cfg["dtype"] == "bf16" else 4
        a = outs[0].long().cpu()
        a = a[a >= 0]
        if mode == "sample_lazy":
            g = cfg["gamma"]
            walk_rows = ((a + 1) + torch.clamp(a + 1, max=g)).sum().item()
            step_rows = walk_rows + torch.where(a < g, 2, 1).sum().item()
        elif mode in ("typical", "onehot"):
            walk_rows = (a + 1).sum().item()
            step_rows = walk_rows + a.numel()
        else:
            walk_rows = step_rows = (a + 1).sum().item()
        lb, sb = walk_rows * cfg["V"] * s, step_rows * cfg["V"] * s
        level = kernel == "level_kernel"
        res.update({"hbm_gbs_step": sb / (ms_step / 1e3) / 1e9, "frac_of_8tbs_step": sb / (ms_step / 1e3) / 8e12,
                    "lazy": ("a level-synchronous walk over the whole GPU reads only the rows the rule needs"
                             if level else "a cluster of CTAs per sequence (one CTA when the batch fills the GPU) "
                             "reads only the rows the rule needs"),
                    "rows_read_per_step": step_rows,
                    "roofline": {"bound": "hbm", "kernel": kernel, "achieved": lb / (dom_ms / 1e3) / 1e9,
                                 "peak": peak, "peak_kind": peak_kind + " copy (read+write) bandwidth",
                                 "unit": "GB/s", "frac": lb / (dom_ms / 1e3) / 1e9 / peak, "bytes_per_launch": lb,
                                 "traffic": committed_traffic(kernel, name),
                                 "note": "bytes the walk needs (a lower bound for tree greedy) over the walk's time"}})
    return res, inputs, call


def measure_e2e(name, inputs, steps, dev, **ov):
    """The same metric through the public call with host buffers: every step copies its
    inputs from pinned host memory and reads the results back."""
    import torch
    from speculative_decoding_verify_spec_gb300 import workloads as W

    cfg = dict(W.WORKLOADS[name])
    cfg.update(ov)
    mode = cfg["mode"]
    host_in = {}
    dev_in = {}
    keys = {"sample": ["target", "draft", "draft_tokens"], "greedy": ["target", "draft_tokens"],
            "tree": ["target", "node_tokens"],
            "tree_sample": ["target", "draft", "node_tokens"], "ngram": ["history", "lengths"]}[mode]
    target_only = bool(cfg.get("typical") or cfg.get("onehot"))  # no draft logits
    if target_only:
        keys = ["target", "draft_tokens"]
    for k in keys:
        t = getattr(inputs, k)
        host_in[k] = t.cpu().pin_memory()
        dev_in[k] = torch.empty_like(t)
    call, outs = make_call(name, inputs, dev, **ov)
    host_out = [o.cpu().pin_memory() for o in outs]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out)

    def step():
        for k in keys:
            dev_in[k].copy_(host_in[k], non_blocking=True)
        if mode == "ngram":
            call(dev_in["history"], dev_in["lengths"])
        elif target_only:
            call(dev_in["target"], dev_in["draft_tokens"])
        elif mode == "sample":
            call(dev_in["target"], dev_in["draft"], dev_in["draft_tokens"])
        elif mode == "greedy":
            call(dev_in["target"], dev_in["draft_tokens"])
        elif mode == "tree_sample":
            call(dev_in["target"], dev_in["node_tokens"], dev_in["draft"])
        else:
            call(dev_in["target"], dev_in["node_tokens"])
        for h, o in zip(host_out, outs):
            h.copy_(o, non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        step()
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    return {"value": cfg["B"] / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def oracle_run(name, inputs, threads, limit=None):
    """The oracle over a batch (its first `limit` sequences if given), one thread per range
    of sequences; returns (sequences, threads used, accepted_len or None, flags or None)."""
    import numpy as np
    import oracle
    from speculative_decoding_verify_spec_gb300 import workloads as W

    cfg = W.WORKLOADS[name]
    mode = cfg["mode"]
    orc = oracle.default()
    if mode == "ngram":
        h = inputs.history.cpu().numpy()
        L = np.clip(inputs.lengths.cpu().numpy(), 0, h.shape[1])
        B = h.shape[0] if limit is None else min(limit, h.shape[0])
        fn = lambda r: orc.ngram_draft(h[r[0]:r[1]], L[r[0]:r[1]], inputs.n, inputs.k, inputs.pad)
    else:
        t = oracle.as_oracle_logits(inputs.target)
        B = t.shape[0] if limit is None else min(limit, t.shape[0])
    step = max(1, (B + threads - 1) // threads)
    ranges = [(s, min(B, s + step)) for s in range(0, B, step)]
    T, seed = getattr(inputs, "temperature", None), getattr(inputs, "seed", None)
    if mode == "sample" and cfg.get("typical"):
        x = inputs.draft_tokens.cpu().numpy()

        def fn(r):
            acc, _, flags, _ = orc.verify_typical(t[r[0]:r[1]], x[r[0]:r[1]], T, cfg["epsilon"], cfg["delta"],
                                                  seed, 0, b0=r[0])
            return acc, flags
    elif mode == "sample" and cfg.get("onehot"):
        x = inputs.draft_tokens.cpu().numpy()
        g, V = x.shape[1], t.shape[2]

        def fn(r):  # q one-hot on each draft token: -inf everywhere else, in the target's form
            n = r[1] - r[0]
            if t.dtype == np.uint16:
                d = np.full((n, g, V), 0xFF80, np.uint16)  # bf16 -inf
            else:
                d = np.full((n, g, V), -np.inf, np.float32)
            if g:
                d[np.arange(n)[:, None], np.arange(g)[None, :], x[r[0]:r[1]]] = 0
            acc, _, flags = orc.verify_sample(t[r[0]:r[1]], d, x[r[0]:r[1]], T, seed, 0, b0=r[0])
            return acc, flags
    elif mode == "sample":
        d = oracle.as_oracle_logits(inputs.draft)
        x = inputs.draft_tokens.cpu().numpy()

        def fn(r):
            acc, _, flags = orc.verify_sample(t[r[0]:r[1]], d[r[0]:r[1]], x[r[0]:r[1]], T, seed, 0, b0=r[0])
            return acc, flags
    elif mode == "greedy":
        x = inputs.draft_tokens.cpu().numpy()
        fn = lambda r: (orc.verify_greedy(t[r[0]:r[1]], x[r[0]:r[1]])[0], None)
    elif mode == "tree_sample":
        d = oracle.as_oracle_logits(inputs.draft)
        par = inputs.parent.cpu().numpy()
        x = inputs.node_tokens.cpu().numpy()

        def fn(r):
            acc, _, _, flags = orc.verify_tree_sample(t[r[0]:r[1]], d[r[0]:r[1]], par, x[r[0]:r[1]],
                                                      inputs.max_depth, T, seed, 0,
                                                      inputs.without_replacement, b0=r[0])
            return acc, flags
    elif mode == "tree":
        par = inputs.parent.cpu().numpy()
        x = inputs.node_tokens.cpu().numpy()

        def fn(r):
            acc, _, _, flags = orc.verify_tree_greedy(t[r[0]:r[1]], par, x[r[0]:r[1]], inputs.max_depth)
            return acc, flags
    with ThreadPoolExecutor(threads) as ex:
        res = list(ex.map(fn, ranges))
    if mode == "ngram" or not res:
        return B, len(ranges), None, None
    acc = np.concatenate([r[0] for r in res])
    flags = np.concatenate([r[1] for r in res]) if res[0][1] is not None else None
    return B, len(ranges), acc, flags


def oracle_acceptance(acc, flags):
    """Accepted-length histogram of an oracle run and how many sequences it flagged as
    decided within its tolerance of a threshold or CDF boundary."""
    import numpy as np

    acc = np.asarray(acc)
    valid = acc[acc >= 0]
    out = {"sequences": int(acc.size), "invalid": int((acc < 0).sum()),
           "accepted_len_hist": [int(x) for x in np.bincount(valid)] if valid.size else [],
           "mean_accepted_len": float(valid.mean()) if valid.size else None}
    if flags is not None:
        n = int((np.asarray(flags) != 0).sum())
        out.update({"oracle_flags": n, "oracle_flag_rate": n / max(1, acc.size)})
    return out


def cpu_baseline(name, inputs):
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()
    B, used, acc, flags = oracle_run(name, inputs, cores)
    dt = time.perf_counter() - t0
    n1 = 16  # and single-threaded, on the batch's first sequences
    t1 = time.perf_counter()
    B1, _, _, _ = oracle_run(name, inputs, 1, limit=n1)
    dt1 = time.perf_counter() - t1
    return {"value": B / dt, "unit": UNIT, "cores": min(cores, used), "kind": "oracle",
            "sample": f"all {B} sequences, once ({dt:.2f} s on {min(cores, used)} threads)",
            "single_thread": {"value": B1 / dt1, "unit": UNIT, "cores": 1,
                              "sample": f"the first {B1} sequences of the batch ({dt1:.2f} s wall)"},
            "acceptance": oracle_acceptance(acc, flags) if acc is not None else None}


def brief(r, full=True):
    """A configuration's headline figures, for the compact final line: seqs/s, ms per step,
    the step's share of 8 TB/s, the dominant kernel's fraction of the measured copy peak and
    its ncu traffic, the CUDA-graph replay time, and marked / redone sequences."""
    rf = r.get("roofline") or {}
    acc = r.get("acceptance") or {}

    def g(x):
        return float(f"{x:.4g}") if isinstance(x, float) else x

    out = {"value": g(r["value"]), "ms": g(r["ms_per_step"]), "frac_8tbs": g(r.get("frac_of_8tbs_step")),
           "roofline_frac": g(rf.get("frac"))}
    if full:
        out.update({"traffic": rf.get("traffic"), "graph_ms": g((r.get("graph") or {}).get("ms_per_step"))})
        if acc.get("redraw_marked") is not None:
            out["redone"] = f"{acc['redraw_redone']}/{acc['redraw_marked']}"
    return {k: v for k, v in out.items() if v is not None}


def compact_line(line, main, modes, workload):
    """The final JSON line: the contract's keys, then every configuration's headline figures
    (C1 .. C5, then the NEXT rules) -- short enough that its whole text survives a tail."""
    keep = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
            "scaling", "vs_baseline", "dtype", "data", "config", "frac_of_8tbs", "roofline", "gpu_launches",
            "clocks")
    out = {k: line[k] for k in keep}
    out["config"] = {k: v for k, v in out["config"].items() if k in ("workload", "l2")}
    if out["roofline"] is not None:
        out["roofline"] = {k: v for k, v in out["roofline"].items() if k != "bytes_per_launch"}
    e2e = line["e2e"]
    out["e2e"] = {k: e2e[k] for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step")}
    cpu = line.get("cpu_baseline")
    out["cpu_baseline"] = None if cpu is None else {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")}
    allr = dict(modes)
    allr[workload] = main
    out["configs"] = {CONFIGS[n]: brief(allr[n]) for n in CONFIGS if n in allr}
    out["next"] = {n: brief(r, full=False) for n, r in modes.items() if n not in CONFIGS}
    return out


def run_ours(args):
    import torch

    rank, world, local = dist_setup("nccl" if args.gpus > 1 else "gloo")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    import __graft_entry__

    __graft_entry__.build()
    from speculative_decoding_verify_spec_gb300 import workloads as W

    peak, peak_kind = hbm_peak()
    clocks = ClockSampler(local)
    clocks.start()
    ov = {} if args.batch is None else {"B": args.batch}
    main, inputs, _ = measure(args.workload, args.steps, args.warmup, rank, world, dev, peak,
                              peak_kind, args.batch, detail=True)
    clk = clocks.stop()
    modes = {}
    if not args.no_modes:
        for name in SECONDARY:
            if name == args.workload:
                continue
            r, inp, _ = measure(name, args.steps, args.warmup, rank, world, dev, peak, peak_kind,
                                args.batch, graph=name == "sample_b1")
            modes[name] = r
            del inp
            torch.cuda.empty_cache()
    e2e = measure_e2e(args.workload, inputs, max(3, args.e2e_steps), dev, **ov)
    e2e_val = max_over_ranks(e2e["ms_per_step"], world, dev)
    e2e["value"] = world * ov.get("B", W.WORKLOADS[args.workload]["B"]) / (e2e_val / 1e3)
    e2e["ms_per_step"] = e2e_val
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload, inputs)
    if rank == 0:
        cfg = dict(W.WORKLOADS[args.workload])
        cfg.update(ov)
        line = {
            "metric": METRIC, "value": main["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": main["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded generators, resident in HBM)",
            "config": {"workload": W.DESCRIPTIONS[args.workload], "B": cfg["B"],
                       "gamma": cfg.get("gamma"), "V": cfg["V"], "logits": cfg.get("dtype"),
                       "temperature": cfg.get("temperature"), "l2": main["l2"],
                       "parallelism": f"replicas x{world} (independent batches per GPU)"},
            "rows_per_s": main["rows_per_s"], "hbm_gbs": main["hbm_gbs_step"],
            "frac_of_8tbs": main["frac_of_8tbs_step"],
            "mean_accepted_len": main["mean_accepted_len"], "acceptance": main.get("acceptance"),
            "stages_ms": main["stages_ms"],
            "step_spread": main.get("step_spread"), "graph": main.get("graph"),
            "roofline": main["roofline"], "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": main["gpu_launches"], "clocks": clk, "modes": modes,
        }
        # every detail on one earlier line (not a JSON line of its own), then the compact line
        print("detail " + json.dumps(line), flush=True)
        print(json.dumps(compact_line(line, main, modes, args.workload)), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ----------------------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ----------------------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    from speculative_decoding_verify_spec_gb300 import workloads as W
    import __graft_entry__

    __graft_entry__._build_oracle()
    name = args.workload
    cfg = W.WORKLOADS[name]
    cores = os.cpu_count() or 1
    per_step = min(cfg["B"], cores)
    inputs = W.make(name, device="cpu", B=per_step)
    for _ in range(max(1, min(args.warmup, 3))):
        oracle_run(name, inputs, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _, _, acc, flags = oracle_run(name, inputs, cores)
    dt = time.perf_counter() - t0
    value = args.steps * per_step / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generators)",
        "config": {"workload": W.DESCRIPTIONS[name], "B": cfg["B"], "gamma": cfg.get("gamma"),
                   "V": cfg["V"], "logits": cfg.get("dtype")},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(cores, per_step), "kind": "oracle",
                         "sample": f"{per_step} sequences of the workload per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "acceptance": oracle_acceptance(acc, flags) if args.steps > 0 and acc is not None else None,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
