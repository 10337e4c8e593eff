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
