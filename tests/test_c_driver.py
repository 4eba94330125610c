"""The C ABI from a plain C program (no Python, no C++, no GPU): tests/c/abi_driver.c is compiled
with the system C compiler against include/k3moe.h, linked to libk3moe.so, and run."""
import os
import shutil
import subprocess

import pytest

import mxfp4_routed_expert_06_b300 as k3

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c_caller(tmp_path):
    libdir = os.path.dirname(k3.LIB_PATH)
    exe = str(tmp_path / "abi_driver")
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(k3.HEADER),
                           os.path.join(HERE, "c", "abi_driver.c"), "-o", exe, "-L", libdir, "-lk3moe",
                           "-Wl,-rpath," + libdir])
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "ok"
