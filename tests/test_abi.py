"""The C-ABI library on the CPU: it loads, exports every declared symbol with C linkage,
and its host-side checks reject bad arguments before touching the GPU.  No compute call
is made here (there may be no GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

from speculative_decoding_verify_spec_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(spec_verify_\w+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    _build.build_library()
    return binding.load_library()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("spec_verify_sample", "spec_verify_greedy", "spec_verify_tree_greedy",
                 "spec_verify_workspace_size", "spec_verify_row_stats",
                 "spec_verify_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.check_output(["nm", "-D", "--defined-only", _build.LIB_PATH]).decode()
    exported = set(re.findall(r"\bT (\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_version_and_status_strings(lib):
    assert lib.spec_verify_version() == 100
    for code in range(6):
        assert lib.spec_verify_status_string(code).decode() not in ("", "unknown status")
    assert lib.spec_verify_status_string(99).decode() == "unknown status"


def test_workspace_sizes(lib):
    ws = lib.spec_verify_workspace_size
    # sampling, B=256, gamma=8, V=128256, bf16: 63 tiles of 2048 logits per row (one
    # partial each) and 126 residual tiles of 1024 (one mass each) on the stop row
    n = ws(0, 256, 8, 128256, 1)
    assert n >= 256 * 17 * 63 * 8 + 256 * 17 * 8 + 256 * 8 + 256 * 126 * 4
    assert n % 256 == 0
    assert ws(1, 512, 6, 152064, 1) >= 512 * 7 * 75 * 8
    assert ws(2, 64, 64, 128256, 1) >= 64 * 64 * 63 * 8
    assert ws(0, 0, 8, 1000, 0) == 0
    assert ws(8, 1, 1, 1, 0) == 0  # an unknown mode
    # the re-draw of every marked sequence: per sequence 5 rows of double-float unit sums and
    # one of counts (64-logit units), plus the control words, marks and 2 B records
    assert n >= 256 * 5 * 2004 * 8 + 256 * 2004 * 4 + 4 * (8 + 256)
    # the status words: every sampling mode (0, 4-7), inside its workspace; none elsewhere
    off = lib.spec_verify_status_offset
    off.restype = ctypes.c_size_t
    none = ctypes.c_size_t(-1).value
    for mode in (0, 4, 5, 6, 7):
        o = off(mode, 64, 8, 32000, 1)
        assert o != none and o % 256 == 0 and o + 4 * (8 + 64) <= ws(mode, 64, 8, 32000, 1)
    for mode in (1, 2, 3, 8):
        assert off(mode, 64, 8, 32000, 1) == none
    assert off(0, 0, 8, 32000, 1) == none and off(0, 4, 8, 0, 1) == none and off(0, 4, 8, 10, 5) == none
    # the lazy walks (chain sampling, typical, one-hot): the sampling layout for their rows
    # (2 gamma + 1, or gamma + 1 target rows), plus the walk's lists and counters; typical
    # acceptance adds one float per tile for the entropy's moment
    assert ws(5, 256, 8, 128256, 1) >= ws(0, 256, 8, 128256, 1) + 4 * 5 * 256
    one_hot = ws(7, 256, 8, 128256, 1)
    assert one_hot >= 256 * 9 * 63 * 8 + 256 * 5 * 2004 * 8
    assert ws(6, 256, 8, 128256, 1) >= one_hot + 256 * 9 * 63 * 4


P = ctypes.c_void_p


def _sample(lib, **kw):
    a = dict(t=P(16), tsb=0, tsr=0, d=P(16), dsb=0, dsr=0, dt=1, B=1, g=1, V=10, x=P(16),
             T=1.0, seed=0, off=0, acc=P(16), out=P(16), ws=P(256), wsb=1 << 20, s=None)
    a.update(kw)
    return lib.spec_verify_sample(a["t"], a["tsb"], a["tsr"], a["d"], a["dsb"], a["dsr"], a["dt"],
                                  a["B"], a["g"], a["V"], a["x"], a["T"], a["seed"], a["off"],
                                  a["acc"], a["out"], a["ws"], a["wsb"], a["s"])


def test_sample_rejects_bad_arguments_before_any_launch(lib):
    assert _sample(lib, B=-1) == 1
    assert _sample(lib, V=0) == 1
    assert _sample(lib, g=-1) == 1
    assert _sample(lib, g=2000) == 1
    assert _sample(lib, T=0.0) == 1
    assert _sample(lib, T=float("nan")) == 1
    assert _sample(lib, T=float("inf")) == 1
    assert _sample(lib, tsr=-5) == 1
    assert _sample(lib, t=None) == 1
    assert _sample(lib, d=None) == 1
    assert _sample(lib, dt=7) == 2
    assert _sample(lib, ws=None) == 5
    assert _sample(lib, wsb=16) == 5
    assert _sample(lib, ws=P(8)) == 5          # misaligned workspace
    assert _sample(lib, B=0) == 0              # empty batch: nothing to do


def test_greedy_and_tree_reject_bad_arguments(lib):
    g = lib.spec_verify_greedy
    assert g(P(16), 0, 0, 1, -1, 2, 5, P(16), P(16), P(16), P(256), 1 << 20, None) == 1
    assert g(P(16), 0, 0, 1, 1, 2, 0, P(16), P(16), P(16), P(256), 1 << 20, None) == 1
    assert g(P(16), 0, 0, 1, 1, 2, 5, None, P(16), P(16), P(256), 1 << 20, None) == 1
    assert g(P(16), 0, 0, 1, 1, 2, 5, P(16), P(16), P(16), P(256), 8, None) == 5
    assert g(P(16), 0, 0, 1, 0, 2, 5, P(16), P(16), P(16), P(256), 1 << 20, None) == 0
    t = lib.spec_verify_tree_greedy
    args = [P(16), 0, 0, 1, 1, 7, 5, P(16), P(16), 2, P(16), P(16), P(16), P(256), 1 << 20, None]
    bad_n = list(args)
    bad_n[5] = 0
    assert t(*bad_n) == 1
    too_many = list(args)
    too_many[5] = 5000
    assert t(*too_many) == 1
    bad_depth = list(args)
    bad_depth[9] = 7      # max_depth must be < N
    assert t(*bad_depth) == 1
    no_parent = list(args)
    no_parent[7] = None
    assert t(*no_parent) == 1


def test_uniform_hook_rejects_bad_purpose(lib):
    assert lib.spec_verify_uniforms(1, 0, 1, 1, 2, P(16), None) == 1
    assert lib.spec_verify_uniforms(1, 0, 0, 4, 0, P(16), None) == 0


def test_binding_refuses_cpu_tensors():
    """No entry has a CPU path: host tensors are refused before the library is called."""
    import torch
    t = torch.zeros(2, 3, 8)
    x = torch.zeros(2, 2, dtype=torch.int32)
    tt = torch.zeros(2, 3, 8)
    par = torch.tensor([-1, 0, 0], dtype=torch.int32)
    tok = torch.zeros(2, 3, dtype=torch.int32)
    calls = [
        lambda: binding.spec_verify_greedy(t, x),
        lambda: binding.spec_verify_sample(t, t[:, :2], x, 1.0, 0),
        lambda: binding.spec_verify_tree_greedy(tt, par, tok, 1),
        lambda: binding.spec_verify_tree_sample(tt, tt, par, tok, 1, 1.0, 0),
        lambda: binding.spec_verify_sample_lazy(t, t[:, :2], x, 1.0, 0),
        lambda: binding.spec_verify_greedy_lazy(t, x),
        lambda: binding.spec_verify_tree_greedy_lazy(tt, par, tok, 1),
        lambda: binding.spec_verify_typical(t, x, 1.0, 0.1, 0.3, 0),
        lambda: binding.spec_verify_sample_onehot(t, x, 1.0, 0),
        lambda: binding.spec_verify_greedy_noalloc(t, x),
        lambda: binding.spec_verify_row_stats(t),
        lambda: binding.spec_ngram_draft(torch.zeros(2, 16, dtype=torch.int32),
                                         torch.full((2,), 16, dtype=torch.int32), 3, 4),
    ]
    for call in calls:
        with pytest.raises(ValueError):
            call()


def test_binding_checks_caller_provided_outputs():
    """Outputs and workspaces passed in are written in place by the kernels, so anything
    but a contiguous int32 tensor of the right shape on the call's device is refused."""
    import torch
    dev = torch.device("cuda", 0)
    with pytest.raises(ValueError):
        binding._out(torch.zeros(4, dtype=torch.int32), "accepted_len", (4,), dev)   # host memory
    assert binding._out(None, "x", (2, 3), torch.device("cpu")).shape == (2, 3)      # allocated when absent
    with pytest.raises(ValueError):
        binding._workspace(binding.MODE_GREEDY, 1, 1, 8, binding.FP32, dev, torch.zeros(1 << 16, dtype=torch.uint8))
    with pytest.raises(ValueError):
        binding._like(torch.zeros(1, 1, 4, dtype=torch.bfloat16), torch.zeros(1, 1, 4), "draft")


def test_tree_sample_and_lazy_entries_reject_bad_arguments(lib):
    ts = lib.spec_verify_tree_sample
    # t tsb tsr d dsb dsr dtype B N V parent tokens max_depth T seed off wr acc out path ws wsb stream
    base = [P(16), 0, 0, P(16), 0, 0, 1, 1, 7, 5, P(16), P(16), 2, 1.0, 0, 0, 1, P(16), P(16), P(16),
            P(256), 1 << 20, None]

    def call(fn, args, **at):
        a = list(args)
        for i, v in at.items():
            a[int(i[1:])] = v
        return fn(*a)
    assert call(ts, base, a6=9) == 2                     # unknown dtype
    assert call(ts, base, a8=0) == 1                     # N < 1
    assert call(ts, base, a8=5000) == 1                  # N above the limit
    assert call(ts, base, a12=7) == 1                    # max_depth must be < N
    assert call(ts, base, a2=-3) == 1                    # negative stride
    assert call(ts, base, a13=0.0) == 1                  # temperature must be > 0
    assert call(ts, base, a13=float("inf")) == 1
    assert call(ts, base, a10=None) == 1                 # no parent array
    assert call(ts, base, a3=None) == 1                  # no draft logits
    assert call(ts, base, a20=None) == 5                 # no workspace
    assert call(ts, base, a7=0) == 0                     # empty batch
    sl = lib.spec_verify_sample_lazy
    # t tsb tsr d dsb dsr dtype B gamma V x T seed off acc out ws wsb stream
    lz = [P(16), 0, 0, P(16), 0, 0, 1, 1, 2, 5, P(16), 1.0, 0, 0, P(16), P(16), P(256), 1 << 20, None]
    assert call(sl, lz, a8=-1) == 1
    assert call(sl, lz, a8=2000) == 1
    assert call(sl, lz, a11=float("nan")) == 1
    assert call(sl, lz, a10=None) == 1                   # drafts needed when gamma > 0
    assert call(sl, lz, a16=P(8)) == 5                   # misaligned workspace
    assert call(sl, lz, a7=0) == 0
    gl = lib.spec_verify_greedy_lazy
    assert gl(P(16), 0, 0, 1, 1, 2, 0, P(16), P(16), P(16), None) == 1      # V < 1
    assert gl(P(16), 0, 0, 1, 1, 2, 5, None, P(16), P(16), None) == 1       # no drafts
    assert gl(P(16), 0, 0, 3, 1, 2, 5, P(16), P(16), P(16), None) == 2      # unknown dtype
    assert gl(P(16), 0, 0, 1, 0, 2, 5, P(16), P(16), P(16), None) == 0
    tl = lib.spec_verify_tree_greedy_lazy
    assert tl(P(16), 0, 0, 1, 1, 7, 5, P(16), P(16), 7, P(16), P(16), P(16), None) == 1  # depth >= N
    assert tl(P(16), 0, 0, 1, 1, 7, 5, None, P(16), 2, P(16), P(16), P(16), None) == 1   # no parent
    assert tl(P(16), 0, 0, 1, 0, 7, 5, P(16), P(16), 2, P(16), P(16), P(16), None) == 0


def test_target_only_rules_reject_bad_arguments(lib):
    ty = lib.spec_verify_typical
    # t tsb tsr dtype B gamma V x T eps delta seed off acc out ws wsb stream
    base = [P(16), 0, 0, 1, 1, 2, 5, P(16), 1.0, 0.1, 0.3, 0, 0, P(16), P(16), P(256), 1 << 20, None]

    def call(fn, args, **at):
        a = list(args)
        for i, v in at.items():
            a[int(i[1:])] = v
        return fn(*a)
    assert call(ty, base, a9=-0.1) == 1                  # epsilon must be >= 0
    assert call(ty, base, a10=float("nan")) == 1         # delta must be finite
    assert call(ty, base, a10=float("inf")) == 1
    assert call(ty, base, a8=0.0) == 1
    assert call(ty, base, a7=None) == 1
    assert call(ty, base, a3=5) == 2
    assert call(ty, base, a16=8) == 5                    # workspace too small
    assert call(ty, base, a4=0) == 0
    oh = lib.spec_verify_sample_onehot
    # t tsb tsr dtype B gamma V x T seed off acc out ws wsb stream
    ob = [P(16), 0, 0, 1, 1, 2, 5, P(16), 1.0, 0, 0, P(16), P(16), P(256), 1 << 20, None]
    assert call(oh, ob, a5=-1) == 1
    assert call(oh, ob, a8=-1.0) == 1
    assert call(oh, ob, a11=None) == 1                   # no accepted_len
    assert call(oh, ob, a13=None) == 5
    assert call(oh, ob, a4=0) == 0


def test_drafter_and_hooks_reject_bad_arguments(lib):
    ng = lib.spec_ngram_draft
    # history stride lengths B n k pad drafts count stream
    assert ng(P(16), 8, P(16), 1, 0, 4, 0, P(16), P(16), None) == 1          # n < 1
    assert ng(P(16), 8, P(16), 1, 3, -1, 0, P(16), P(16), None) == 1         # k < 0
    assert ng(P(16), -8, P(16), 1, 3, 4, 0, P(16), P(16), None) == 1         # negative stride
    assert ng(P(16), 8, None, 1, 3, 4, 0, P(16), P(16), None) == 1           # no lengths
    assert ng(P(16), 8, P(16), 1, 3, 4, 0, None, P(16), None) == 1           # drafts needed when k > 0
    assert ng(P(16), 8, P(16), 0, 3, 4, 0, P(16), P(16), None) == 0          # empty batch
    rs = lib.spec_verify_row_stats
    assert rs(P(16), 0, 0, 1, 1, 0, 5, 1.0, P(16), P(16), P(256), 1 << 20, None) == 1   # rows < 1
    assert rs(P(16), 0, 0, 1, 1, 1, 5, 0.0, P(16), P(16), P(256), 1 << 20, None) == 1   # T = 0
    assert rs(P(16), 0, 0, 1, 1, 1, 5, 1.0, None, P(16), P(256), 1 << 20, None) == 1    # no output
    assert rs(P(16), 0, 0, 4, 1, 1, 5, 1.0, P(16), P(16), P(256), 1 << 20, None) == 2
    assert rs(P(16), 0, 0, 1, 0, 1, 5, 1.0, P(16), P(16), P(256), 1 << 20, None) == 0
    assert lib.spec_verify_exp_df(P(16), P(16), -1, P(16), P(16), None) == 1
    assert lib.spec_verify_exp_df(None, None, 0, None, None, None) == 0
    assert lib.spec_verify_exp_df(None, P(16), 4, P(16), P(16), None) == 1
    assert lib.spec_verify_wait_selftest(None, 1, 1000, None) == 1
    assert lib.spec_verify_wait_selftest(P(16), 0, 1000, None) == 1          # at least one arrival
    assert lib.spec_verify_wait_selftest(P(16), 3, 1000, None) == 1          # at most two
    assert lib.spec_verify_wait_selftest(P(16), 2, 6_000_000, None) == 1     # limit above 5 s
    assert lib.spec_verify_set_stage_events(None, -1) == 1
    assert lib.spec_verify_set_stage_events(None, 9) == 1
    assert lib.spec_verify_set_stage_events(None, 0) == 0                    # clears the list


def test_binding_constants_match_the_header():
    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "spec_verify.h")).read(), flags=re.S)
    values = {k: int(v) for k, v in re.findall(r"\b(SV_[A-Z0-9_]+)\s*=\s*(\d+)", text)}
    assert values["SV_OK"] == binding.SV_OK
    assert (values["SV_FP32"], values["SV_BF16"]) == (binding.FP32, binding.BF16)
    for name in ("SAMPLE", "GREEDY", "TREE", "ROW_STATS", "TREE_SAMPLE", "SAMPLE_LAZY", "TYPICAL",
                 "SAMPLE_ONEHOT"):
        assert values["SV_MODE_" + name] == getattr(binding, "MODE_" + name), name
    assert values["SV_ERR_TIMEOUT"] == 4  # the status the bounded-wait test expects


def test_package_exports_every_entry_point():
    import speculative_decoding_verify_spec_gb300 as sv
    public = [n for n in dir(binding) if n.startswith(("spec_verify_", "spec_ngram_"))
              and n not in ("spec_verify_exp_df", "spec_verify_uniforms")]
    hooks = {"spec_verify_exp_df"}  # test hooks stay in the binding module
    for n in public:
        assert n in sv.__all__ or n in hooks, n
    for n in sv.__all__:
        assert hasattr(sv, n), n


def test_product_build_has_no_check_word(lib):
    info = (ctypes.c_int32 * 4)(7, 7, 7, 7)
    assert lib.spec_verify_check_word(info) == 2  # SV_ERR_UNSUPPORTED, no device access
    assert list(info) == [0, 0, 0, 0]
    assert lib.spec_verify_check_word(None) == 2
    assert lib.spec_verify_check_selftest(ctypes.c_int64(5), ctypes.c_int64(3)) == 2
    assert lib.spec_verify_status_string(6) == b"an internal index left its extent (bounds-checked build)"


def test_file_tags_follow_fnv1a():
    # FNV-1a (32-bit) reference values: "" -> 0x811c9dc5, "a" -> 0xe40c292c, "foobar" -> 0xbf9cf968
    fold = lambda h: (h >> 16) ^ (h & 0xFFFF)
    assert binding.file_tag("") == fold(0x811C9DC5)
    assert binding.file_tag("a") == fold(0xE40C292C)
    assert binding.file_tag("foobar") == fold(0xBF9CF968)
    names = [f for f in os.listdir(os.path.join(_build.CSRC)) if f.endswith((".cu", ".cuh"))]
    assert len({binding.file_tag(f) for f in names}) == len(names)  # the tags tell the files apart
