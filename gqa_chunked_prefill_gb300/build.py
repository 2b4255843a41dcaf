"""Builds libgqa_prefill.so in-tree with nvcc for sm_103a (no torch, no cmake).

Each .cu translation unit is compiled in parallel, then linked into one shared
library with the CUDA runtime linked statically, so the library loads on a
machine without a GPU (it only needs the driver once a CUDA call is made).
"""
from __future__ import annotations

import os
import platform
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libgqa_prefill.so")
CHECKED_LIB = os.path.join(PKG, "libgqa_prefill_checked.so")  # built with GQA_CHECK_BOUNDS

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _arch_matches(stamp: str) -> bool:
    try:
        return open(stamp).read().strip() == platform.machine()
    except OSError:
        return False


def build(force: bool = False, verbose: bool = False, extra_flags=(), check_bounds: bool = False) -> str:
    """libgqa_prefill.so, or with check_bounds the bounds-checked libgqa_prefill_checked.so
    (same sources and ABI; every epilogue store and merge access checks its row)."""
    lib = CHECKED_LIB if check_bounds else LIB
    build_dir = os.path.join(PKG, "_build", platform.machine() + ("-checked" if check_bounds else ""))
    stamp = lib + ".arch"
    if check_bounds:
        extra_flags = list(extra_flags) + ["-DGQA_CHECK_BOUNDS=1"]
    os.makedirs(build_dir, exist_ok=True)
    force = force or not _arch_matches(stamp)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    objs, jobs = [], []
    for src in sources():
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            jobs.append([nvcc(), *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed: " + " ".join(cmd))

    with ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(lib, objs):
        run([nvcc(), *ARCH, "-shared", "-o", lib + ".tmp", *objs])
        os.replace(lib + ".tmp", lib)
        with open(stamp, "w") as f:
            f.write(platform.machine())
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []))
