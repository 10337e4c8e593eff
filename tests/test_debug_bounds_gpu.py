"""The address-checking build (GDN_DEBUG_BOUNDS): every computed global index of the verify,
commit and attention kernels is checked against its array before the access, and a violation sets
GDN_STATUS_OUT_OF_BOUNDS instead of touching memory. It stands in for a memory checker.

The test loads that build (GDN_TREE_DEBUG_BOUNDS=1) in a child process and runs the small cases of
the parity suites through it; those tests require status 0 and oracle parity, so an index the
checks reject fails them. No case is built to go out of bounds.
"""

import os
import subprocess
import sys

import pytest

from gated_deltanet_tree_03_b300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu

SMALL_CASES = [
    "tests/test_parity_gpu.py::test_chain3_d32_full",
    "tests/test_parity_gpu.py::test_random_ragged_trees",
    "tests/test_parity_gpu.py::test_extreme_shapes",
    "tests/test_parity_gpu.py::test_small_trees_streaming_kernel",
    "tests/test_parity_gpu.py::test_mixed_key_value_widths",
    "tests/test_parity_gpu.py::test_rootbranch6_full",
    "tests/test_serving_gpu.py",
    "tests/test_commit_verify_gpu.py",
    "tests/test_attention_gpu.py",
]


def _env():
    env = dict(os.environ)
    env["GDN_TREE_DEBUG_BOUNDS"] = "1"
    return env


def test_debug_build_is_loaded():
    _build.build(debug_bounds=True)
    code = "from gated_deltanet_tree_03_b300 import binding as gb; print(gb.library()._name)"
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=_env(), capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip().endswith("libgdn_tree_debug_bounds.so")


def test_small_parity_cases_pass_with_address_checks():
    _build.build(debug_bounds=True)
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *SMALL_CASES]
    r = subprocess.run(cmd, cwd=ROOT, env=_env(), capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
