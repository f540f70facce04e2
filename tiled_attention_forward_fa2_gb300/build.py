"""Build the CUDA library in-tree: lib/libattn_fwd_gb300.so for sm_103a.

nvcc compiles csrc/attn_fwd.cu (host launcher + kernels) with the static CUDA
runtime, so the library loads without a GPU driver (the C ABI can then still
validate arguments) and links no libcuda: tensor maps are encoded through the
runtime's driver entry point.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libattn_fwd_gb300.so")
# The same sources with -DATTN_TEST_HOOKS: adds attn_test_withhold_kv, which
# makes the forward drop its K/V loads (to drive the timeout path).  Only the
# failure-detection tests load it; the production library cannot do this.
LIB_TEST = os.path.join(LIBDIR, "libattn_fwd_gb300_testhooks.so")
SOURCES = [os.path.join(CSRC, "attn_fwd.cu")]  # includes the backward (one module, one status word)
DEPS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")] + \
    [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return exe


def stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(d) > t for d in DEPS)


def _command(out: str, defines) -> list:
    return [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-I" + INCLUDE,
            *defines, "-Xptxas", "-v", "-o", out, *SOURCES]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the production library and its test-hook variant (in parallel) if
    missing or older than their sources; returns the production library's path."""
    os.makedirs(LIBDIR, exist_ok=True)
    jobs = []
    for lib, defines in ((LIB, []), (LIB_TEST, ["-DATTN_TEST_HOOKS"])):
        if force or stale(lib):
            tmp = lib + f".tmp{os.getpid()}"
            proc = subprocess.Popen(_command(tmp, defines), stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
            jobs.append((lib, tmp, proc))
    errors = []
    for lib, tmp, proc in jobs:
        out, err = proc.communicate()
        if proc.returncode != 0:
            errors.append(f"nvcc failed for {os.path.basename(lib)}:\n{out}{err}")
            continue
        if verbose and lib == LIB:
            print(err)
        os.replace(tmp, lib)
    if errors:
        raise RuntimeError("\n".join(errors))
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
