"""The C ABI from a plain C program: tests/c_abi_consumer.c is compiled with gcc against
include/gdn_tree.h, linked to the built library and run. It needs no GPU (every call it makes
returns before touching CUDA)."""

import os
import shutil
import subprocess

import pytest

from gated_deltanet_tree_03_b300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_plain_c_program_uses_the_library(tmp_path):
    lib = _build.build()
    exe = tmp_path / "c_abi_consumer"
    src = os.path.join(ROOT, "tests", "c_abi_consumer.c")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", f"-I{_build.INCLUDE}", src, "-o", str(exe), lib,
                    f"-Wl,-rpath,{os.path.dirname(lib)}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "ok"


def _build_host_cost(tmp_path):
    lib = _build.build()
    exe = tmp_path / "c_abi_host_cost"
    src = os.path.join(ROOT, "tests", "c_abi_host_cost.c")
    cuda = "/usr/local/cuda"
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-Werror", f"-I{_build.INCLUDE}", f"-I{cuda}/include", src,
                    "-o", str(exe), lib, f"-L{cuda}/lib64", "-lcudart", f"-Wl,-rpath,{os.path.dirname(lib)}",
                    f"-Wl,-rpath,{cuda}/lib64"], check=True)
    return exe


@pytest.mark.skipif(shutil.which("gcc") is None or not os.path.isdir("/usr/local/cuda/include"),
                    reason="no C compiler or CUDA headers")
def test_host_cost_program_compiles(tmp_path):
    assert _build_host_cost(tmp_path).exists()


@pytest.mark.gpu
def test_host_cost_per_call_from_c(tmp_path):
    """Per-call host cost of verify and commit, measured from C: after the first call on a device
    the library reuses the device's properties and each kernel's shared-memory limit, so a call
    is argument checks, tensor-map encoding (tensor-core kernel) and the launch."""
    import json
    exe = _build_host_cost(tmp_path)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    rows = [json.loads(line) for line in out.stdout.splitlines() if line.startswith("{")]
    assert [r["shape"] for r in rows] == ["rootbranch6_B1", "chain32_B1"]
    for r in rows:
        print(r)
        assert r["host_us_verify"] < 25.0 and r["host_us_commit"] < 25.0, r
