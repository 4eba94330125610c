"""The library's host code under AddressSanitizer and UndefinedBehaviorSanitizer.

libk3moe_san.so is the library with its host code (argument checks, workspace and cache
bookkeeping, the cache simulator) built with -fsanitize=address,undefined; tests/c/host_san_driver.c,
a plain C program built the same way, drives it.  Without a GPU the driver runs the simulator and
the refusals; with one it also runs a layer in cache mode (evictions, an injected copy failure, a
move to another cache), which exercises the LRU bookkeeping of the miss path."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))


def _build_and_run(tmp_path):
    sys.path.insert(0, os.path.join(ROOT, "mxfp4_routed_expert_06_b300"))
    import importlib.util
    spec = importlib.util.spec_from_file_location("k3moe_build", os.path.join(ROOT, "mxfp4_routed_expert_06_b300",
                                                                               "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    lib = mod.build(sanitize=True)
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "host_san_driver")
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-g", "-fsanitize=address,undefined",
                           "-fno-sanitize-recover=all", "-I", os.path.join(ROOT, "include"),
                           os.path.join(HERE, "c", "host_san_driver.c"), "-o", exe, "-L", libdir, "-lk3moe_san",
                           "-Wl,-rpath," + libdir])
    env = dict(os.environ)
    # CUDA maps memory where ASan keeps its shadow gap; leaks of the CUDA runtime are not ours
    env["ASAN_OPTIONS"] = "protect_shadow_gap=0:detect_leaks=0:abort_on_error=1"
    env["UBSAN_OPTIONS"] = "print_stacktrace=1:halt_on_error=1"
    return subprocess.run([exe], capture_output=True, text=True, timeout=600, env=env)


@pytest.mark.skipif(shutil.which("gcc") is None or shutil.which("nvcc") is None, reason="no compilers")
def test_host_code_under_sanitizers(tmp_path):
    out = _build_and_run(tmp_path)
    assert out.returncode == 0, out.stderr[-4000:]
    assert out.stdout.strip() in ("ok cpu", "ok gpu")


@pytest.mark.gpu
def test_cache_bookkeeping_under_sanitizers_on_gpu(tmp_path):
    out = _build_and_run(tmp_path)
    assert out.returncode == 0, out.stderr[-4000:]
    assert out.stdout.strip() == "ok gpu"
