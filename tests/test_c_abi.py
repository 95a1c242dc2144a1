"""The C ABI from a plain C11 caller (tests/c_abi/abi_demo.c), compiled with gcc against
include/zero.h and linked with libzero.so and the CUDA runtime, as a C user builds it:
host-only calls and error codes on the CPU; two shard steps (one skipped on an inf) and
the ZeRO-3 gather on the GPU."""
import os
import subprocess

import pytest

from sharded_emulated_reduce_gb300 import build as zbuild

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def demo(tmp_path) -> str:
    lib = zbuild.build()
    pkg = os.path.dirname(lib)
    cuda = zbuild.cuda_home()
    exe = str(tmp_path / "abi_demo")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), os.path.join(HERE, "c_abi", "abi_demo.c"),
           "-L", pkg, "-lzero", "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
           f"-Wl,-rpath,{pkg}:{os.path.join(cuda, 'lib64')}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def run(exe, mode):
    r = subprocess.run([exe, mode], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_c_caller_host_only_calls(tmp_path):
    run(demo(tmp_path), "cpu")


@pytest.mark.gpu
def test_c_caller_steps_and_gathers(tmp_path):
    run(demo(tmp_path), "gpu")
