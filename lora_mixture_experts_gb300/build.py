"""Builds libmoelora.so (CUDA for sm_103a) in-tree with nvcc.

The translation units compile in parallel, then link into one shared
library at ``lora_mixture_experts_gb300/_build/libmoelora.so``.  Nothing is
installed outside the repository.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmoelora.so")
# the same library with the kernels' device-side bounds checks compiled in
# (-DMOELORA_DEVICE_CHECKS): a debug build, used by the tests
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(BUILD_CHECKED, "libmoelora_checked.so")
SOURCES = ["align_kernels.cu", "gemm_tc.cu", "moelora_api.cu", "align_noalloc.cu", "merge.cu"]
HEADERS = ["common.cuh", "align.cuh", "gemm_tc.cuh", "merge.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _cuda_home(nvcc):
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _stale(obj, src):
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [src] + [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "moelora.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, extra_flags=None, checked: bool = False) -> str:
    """Compile (if stale) and link the library; returns its path.  checked:
    the debug build with device-side bounds checks, in its own folder."""
    nvcc = _nvcc()
    cuda_home = _cuda_home(nvcc)
    build_dir, lib = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
                    "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    if extra_flags:
        flags += list(extra_flags)
    if checked:
        flags += ["-DMOELORA_DEVICE_CHECKS"]
    procs = []
    objs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(build_dir, s.replace(".cu", ".o"))
        objs.append(obj)
        if _stale(obj, src):
            cmd = [nvcc] + flags + ["-c", src, "-o", obj]
            if verbose:
                print(" ".join(cmd), flush=True)
            procs.append((s, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for s, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            sys.stdout.write(out.decode(errors="replace"))
        if p.returncode:
            failed.append(s)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    if procs or not os.path.exists(lib):
        cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", lib + ".tmp"] + objs + [
            "-Xlinker", "-rpath," + os.path.join(cuda_home, "lib64")]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.run(cmd, check=True)
        os.replace(lib + ".tmp", lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
