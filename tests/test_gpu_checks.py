"""The small and edge-case parity tests, run again against the bounds-checked build of the
library (compiled with -DSV_CHECKS): every index into a buffer the library sizes itself is
checked against its extent, and each test ends by asserting that no check fired (the
autouse fixture in conftest.py).  This is the stand-in for a memory checker."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FILES = ["test_gpu_checks.py", "test_gpu_sample.py", "test_gpu_greedy.py", "test_gpu_lazy.py", "test_gpu_tree_sample.py",
         "test_gpu_typical.py", "test_gpu_onehot.py", "test_gpu_ngram.py", "test_gpu_redraw_all.py",
         "test_zz_no_alloc.py"]
# the full-size workloads and the long statistical runs stay with the product build
SELECT = ("not full_size and not disagreements and not test_workload and not many_rounds "
          "and not exp_df_matches and not under_the_bounds_checked_build")


@pytest.mark.gpu
def test_small_and_edge_cases_under_the_bounds_checked_build():
    from speculative_decoding_verify_spec_gb300 import _build
    path = _build.build_library(checks=True)
    env = dict(os.environ, SV_LIBRARY=path, SV_CHECKS_ASSERT="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "gpu",
                        "-k", SELECT, *[os.path.join("tests", f) for f in FILES]],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = (r.stdout[-4000:] + "\n" + r.stderr[-2000:]).strip()
    print(r.stdout[-600:])
    assert r.returncode == 0, tail
    summary = r.stdout.strip().splitlines()[-1]
    assert " passed" in summary and int(summary.split(" passed")[0].split()[-1]) >= 30, tail


@pytest.mark.gpu
def test_the_checked_build_records_and_reports_a_violation():
    from speculative_decoding_verify_spec_gb300 import binding
    if not os.environ.get("SV_CHECKS_ASSERT"):
        pytest.skip("runs inside the bounds-checked run above")
    assert binding.check_word() == (0, [0, 0, 0, 0])
    assert binding.check_selftest(5, 3) == 0
    assert binding.check_selftest(-1, 3) == 0  # a second violation: counted, the first one kept
    st, info = binding.check_word()
    assert st == 6 and info[1:] == [5, 3, 2]  # SV_ERR_CHECK: index 5 outside [0, 3), 2 violations
    assert (info[0] & 0xFFFFFFFF) >> 16 == binding.file_tag("sv_api.cu")
    assert binding.check_word() == (0, [0, 0, 0, 0])  # read and cleared


@pytest.mark.gpu
def test_the_checked_build_reports_its_word_and_the_product_build_does_not():
    from speculative_decoding_verify_spec_gb300 import binding
    if os.environ.get("SV_LIBRARY"):
        pytest.skip("runs against the product library")
    st, info = binding.check_word()
    assert st == 2 and info == [0, 0, 0, 0]  # SV_ERR_UNSUPPORTED: the product build has no checks
