"""Build libzero.so in place: CUDA kernels for sm_103a plus the C++ host side.

Run ``python -m sharded_emulated_reduce_gb300.build`` (or call :func:`build`). The
translation units compile in parallel; the library is rebuilt only when a source or
header is newer than it. ``build(checked=True)`` (``--checked``) builds the
bounds-checked variant, ``libzero_checked.so``, for tests (see ``zero_bounds_check``).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libzero.so")
BUILD_DIR = os.path.join(HERE, "_build")
CHECKED_LIB = os.path.join(HERE, "libzero_checked.so")
CHECKED_BUILD_DIR = os.path.join(HERE, "_build_checked")

CU_SOURCES = ["step_kernels.cu", "gather_kernel.cu", "noalloc.cu", "selftest.cu"]
CPP_SOURCES = ["plan.cpp"]
HEADERS = [os.path.join(CSRC, "internal.h"), os.path.join(CSRC, "bulk_async.h"),
           os.path.join(CSRC, "grid_sync.h"), os.path.join(CSRC, "bounds.h"),
           os.path.join(ROOT, "include", "zero.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# --fmad=false: no multiply-add contraction anywhere, so every fp32/fp64 operation is
# the single IEEE operation written in the source
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "--fmad=false", "-Xcompiler", "-fPIC",
                     "-I" + os.path.join(ROOT, "include")]


def cuda_home() -> str:
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd: list[str]) -> None:
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        raise RuntimeError(f"compile failed: {os.path.basename(cmd[-1])}")


def build(verbose: bool = False, extra_nvcc: list[str] | None = None,
          checked: bool = False) -> str:
    """Compile libzero.so (with checked, the bounds-checked libzero_checked.so) if needed
    and return its path."""
    lib_path = CHECKED_LIB if checked else LIB
    build_dir = CHECKED_BUILD_DIR if checked else BUILD_DIR
    extra = list(extra_nvcc or []) + (["-DZERO_BOUNDS_CHECK"] if checked else [])
    sources = [os.path.join(CSRC, s) for s in CU_SOURCES + CPP_SOURCES]
    if not _stale(lib_path, sources + HEADERS + [os.path.abspath(__file__)]) and not extra_nvcc:
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    home = cuda_home()
    inc = os.path.join(home, "include")
    jobs = []
    objs = []
    for s in CU_SOURCES:
        obj = os.path.join(build_dir, s + ".o")
        objs.append(obj)
        jobs.append(["nvcc"] + NVCC_FLAGS + extra + ["-c", "-o", obj, os.path.join(CSRC, s)])
    for s in CPP_SOURCES:
        obj = os.path.join(build_dir, s + ".o")
        objs.append(obj)
        jobs.append(["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-I" + inc,
                     "-I" + os.path.join(ROOT, "include"), "-c", "-o", obj,
                     os.path.join(CSRC, s)])
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        list(ex.map(_run, jobs))
    lib64 = os.path.join(home, "lib64")
    tmp = lib_path + ".tmp"
    _run(["nvcc"] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs +
         ["-Xlinker", "-rpath=" + lib64])
    os.replace(tmp, lib_path)
    if verbose:
        print("built", lib_path)
    return lib_path


if __name__ == "__main__":
    build(verbose=True, checked="--checked" in sys.argv[1:])
