"""Shared pytest configuration: the ``gpu`` marker and the repository root on sys.path."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True)
def _bounds_checked_build():
    """Under the bounds-checked library (SV_CHECKS_ASSERT set, SV_LIBRARY naming it), every
    test ends by reading the library's violation word: any index outside its extent fails
    the test, naming the source file, line, index and extent."""
    yield
    if not os.environ.get("SV_CHECKS_ASSERT"):
        return
    from speculative_decoding_verify_spec_gb300 import binding
    if binding._lib is None:  # the test never loaded the library
        return
    st, info = binding.check_word()
    if st == 0:
        return
    csrc = os.path.join(ROOT, "speculative_decoding_verify_spec_gb300", "csrc")
    names = {binding.file_tag(f): f for f in os.listdir(csrc)}
    site = info[0] & 0xFFFFFFFF
    pytest.fail(f"bounds check (status {st}): {names.get(site >> 16, hex(site >> 16))}:{site & 0xFFFF} "
                f"index {info[1]} outside [0, {info[2]}) ({info[3]} violations)")
