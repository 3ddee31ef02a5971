"""The C ABI from plain C: tests/c/abi_host.c compiles against include/cpkv.h
(as C, not C++), links libcpkv.so and exercises the host entry points.  CPU
only: nothing here launches a kernel."""
import os
import subprocess

import pytest

from paged_kv_cache_compose_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_program_uses_the_abi(tmp_path):
    lib = cuda_build.build()
    exe = str(tmp_path / "abi_host")
    cmd = ["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "abi_host.c"), "-o", exe, "-L", os.path.dirname(lib), "-lcpkv",
           "-Wl,-rpath," + os.path.dirname(lib)]
    subprocess.run(cmd, check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "FAIL" not in r.stdout
    assert r.stdout.count("ok ") >= 15
