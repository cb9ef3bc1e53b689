"""The index-checking debug build over the parity suite.

compute-sanitizer is not available, so the library has a debug build
(``build.py --debug`` -> libsplitkv_debug.so, compiled with SKV_DEBUG): every
kernel checks the indices it computes before it uses them (partial slots
written and read, queue ranges, output rows, the planner's scatter
positions), counts a failed check in the plan header and skips the access.
This test builds it and runs the parity, mask-variant and planner suites
against it in a child process (SPLITKV_DEBUG=1 selects the library at
import); every parity comparison and every plan check there also asserts
that the kernels counted no failed check. The parity bounds are the same.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_suite_under_the_index_checking_build():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "block_sparse_cross_gb300", "build.py"),
                        "--debug"], capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, (r.stdout + r.stderr)[-3000:]
    assert r.stdout.strip().endswith("libsplitkv_debug.so")
    env = dict(os.environ, SPLITKV_DEBUG="1")
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "gpu",
         "tests/test_gpu_parity.py", "tests/test_gpu_masks.py", "tests/test_gpu_plan.py",
         "-k", "not config3_full and not large_configs"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=3600)
    tail = (r.stdout + r.stderr)[-4000:]
    assert r.returncode == 0, tail
    assert " passed" in tail and "failed" not in tail, tail
