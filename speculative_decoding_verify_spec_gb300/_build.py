"""Build libspecverify.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each .cu translation unit is compiled in its own nvcc process (in parallel) and the
objects are linked into one shared library with the CUDA runtime linked statically.

The bounds-checked variant (build_library(checks=True)) is the same sources compiled with
-DSV_CHECKS as relocatable device code (its device-side error word is shared by every
translation unit), linked into libspecverify_checks.so beside the product library.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libspecverify.so")
CHECKS_LIB_PATH = os.path.join(PKG, "libspecverify_checks.so")
OBJ_DIR = os.path.join(ROOT, "_build")
CHECKS_FLAGS = ["-DSV_CHECKS", "-rdc=true"]
SOURCES = ["sv_api.cu", "sv_sample.cu", "sv_greedy.cu", "sv_refine.cu", "sv_tree_sample.cu", "sv_tree_refine.cu",
           "sv_lazy.cu", "sv_ngram.cu", "sv_noalloc.cu", "sv_level.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecverify")
    return cand


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "spec_verify.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build_library(force: bool = False, verbose: bool = False, extra_flags=(), checks: bool = False) -> str:
    """Compile and link libspecverify.so (with checks: libspecverify_checks.so); returns its path."""
    lib_path = CHECKS_LIB_PATH if checks else LIB_PATH
    if not force and up_to_date(lib_path):
        return lib_path
    nvcc = _nvcc()
    obj_dir = os.path.join(OBJ_DIR, "checks") if checks else OBJ_DIR
    os.makedirs(obj_dir, exist_ok=True)
    variant = CHECKS_FLAGS if checks else []
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *variant, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd))
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((cmd, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"))
    if failed:
        msg = "\n".join(f"$ {' '.join(c)}\n{o}" for c, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = lib_path + ".tmp"
    link = [nvcc, *ARCH, *(["-rdc=true"] if checks else []), "-shared", "-o", tmp, *objs]
    subprocess.check_call(link)
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
