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
    # the re-walk / re-draw bookkeeping offsets: modes 4-7 only, inside their workspaces
    off = lib.spec_verify_walk_redraw_offset
    off.restype = ctypes.c_size_t
    none = ctypes.c_size_t(-1).value
    for mode in (4, 5, 6, 7):
        o = off(mode, 64, 8, 32000, 1)
        assert o != none and o % 256 == 0 and o + 4 * (8 + 2 * 64) <= ws(mode, 64, 8, 32000, 1)
    for mode in (0, 1, 2, 3, 8):
        assert off(mode, 64, 8, 32000, 1) == none
    # typical acceptance / one-hot sampling: 4 bytes per residual unit per sequence, plus the
    # double-float re-draw scratch (the stop rows' exponentials: 8 slots x 2 rows x V x 8 B)
    assert ws(6, 256, 8, 128256, 1) == ws(7, 256, 8, 128256, 1) >= 256 * 126 * 4 + 8 * 2 * 128256 * 8


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
    import torch
    t = torch.zeros(1, 2, 8)
    with pytest.raises(ValueError):
        binding.spec_verify_greedy(t, torch.zeros(1, 1, dtype=torch.int32))
