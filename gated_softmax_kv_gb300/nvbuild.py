"""Build the CUDA library (libcsa_compress.so) for sm_103a, in-tree, plus the
small libcsa_selftest.so that exposes device helpers to the GPU tests.

Each translation unit under csrc/ is compiled by its own nvcc process (in
parallel), then linked into gated_softmax_kv_gb300/_build/libcsa_compress.so
against the shared CUDA runtime. No torch, cmake or setuptools involved.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libcsa_compress.so")
SELFTEST_SRC = os.path.join(CSRC, "selftest", "csa_selftest.cu")
SELFTEST_LIB = os.path.join(BUILD, "libcsa_selftest.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "-cudart", "shared", f"-I{INCLUDE}", f"-I{CSRC}"]

_lock = threading.Lock()


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcsa_compress.so")
    return path


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__), SELFTEST_SRC]


def stale() -> bool:
    if not (os.path.exists(LIB) and os.path.exists(SELFTEST_LIB)):
        return True
    t = min(os.path.getmtime(LIB), os.path.getmtime(SELFTEST_LIB))
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library if it is missing or older than its sources."""
    with _lock:
        if not (force or stale()):
            return LIB
        os.makedirs(BUILD, exist_ok=True)
        cc = nvcc()
        extra = ["-Xptxas", "-v"] if verbose else []
        procs = []
        objs = []
        for src in sources():
            obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
            objs.append(obj)
            cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                                text=True)))
        st_tmp = SELFTEST_LIB + f".tmp{os.getpid()}"
        cmd = [cc, *ARCH, *NVCC_FLAGS, "-shared", SELFTEST_SRC, "-o", st_tmp]
        procs.append((SELFTEST_SRC, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                     stderr=subprocess.STDOUT, text=True)))
        failed = []
        for src, pr in procs:
            out, _ = pr.communicate()
            if verbose or pr.returncode != 0:
                sys.stderr.write(out)
            if pr.returncode != 0:
                failed.append(src)
        if failed:
            raise RuntimeError(f"nvcc failed on {', '.join(os.path.basename(f) for f in failed)}")
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run([cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs], check=True)
        os.replace(tmp, LIB)
        os.replace(st_tmp, SELFTEST_LIB)
        return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
