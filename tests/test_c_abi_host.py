"""The C ABI used from C: tests/c_abi/abi_host.c compiles as C99 against
include/prism.h, links libprism.so and checks the host-side entry points
(plan sizes of the 2K-like grid, rejections, trace setter).  No GPU needed."""
import os
import shutil
import subprocess

import pytest

from content_adaptive_block_02_b300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not installed")
def test_host_entry_points_from_c(tmp_path):
    build.build()
    lib_dir = os.path.dirname(build.LIB)
    exe = tmp_path / "abi_host"
    cuda_lib = "/usr/local/cuda/lib64"
    cmd = ["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi", "abi_host.c"), "-o", str(exe),
           "-L", lib_dir, "-lprism", "-Wl,-rpath," + lib_dir]
    if os.path.isdir(cuda_lib):
        cmd += ["-Wl,-rpath," + cuda_lib]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ)
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
