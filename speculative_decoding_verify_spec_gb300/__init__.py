"""GB300-native speculative-decoding verification step.

The product is the C-ABI library ``libspecverify.so`` (hand-written sm_103a CUDA kernels,
declared in ``include/spec_verify.h``).  This package holds its sources (``csrc/``), the
in-tree build (``_build``), the ctypes binding (``binding``) and the seeded input
generators shared by tests and bench (``workloads``).
"""
from .binding import (  # noqa: F401
    SpecVerifyError,
    load_library,
    spec_ngram_draft,
    spec_verify_greedy,
    spec_verify_greedy_lazy,
    spec_verify_typical,
    spec_verify_sample_onehot,
    spec_verify_row_stats,
    spec_verify_sample,
    spec_verify_sample_lazy,
    spec_verify_tree_greedy,
    spec_verify_tree_greedy_lazy,
    spec_verify_tree_sample,
    spec_verify_uniforms,
    spec_verify_workspace_size,
)

__all__ = [
    "SpecVerifyError",
    "load_library",
    "spec_ngram_draft",
    "spec_verify_greedy",
    "spec_verify_greedy_lazy",
    "spec_verify_typical",
    "spec_verify_sample_onehot",
    "spec_verify_row_stats",
    "spec_verify_sample",
    "spec_verify_sample_lazy",
    "spec_verify_tree_greedy",
    "spec_verify_tree_greedy_lazy",
    "spec_verify_tree_sample",
    "spec_verify_uniforms",
    "spec_verify_workspace_size",
]
