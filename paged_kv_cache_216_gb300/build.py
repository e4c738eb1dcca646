"""Build libpa.so (the C ABI of include/pa.h) in-tree for sm_103a.

    python -m paged_kv_cache_216_gb300.build [--force]

Each CUDA translation unit is compiled by nvcc for
``-gencode arch=compute_103a,code=sm_103a``, host C++ by g++, all in
parallel, then linked into ``paged_kv_cache_216_gb300/_build/libpa.so``.
ptxas register/spill reports go to ``_build/ptxas.log``.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libpa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "-I" + INCLUDE, "-I" + CSRC]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall", "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpa.so")


def _cuda_include() -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(_nvcc()))), "include")


def sources():
    cu = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))
    cpp = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cpp"))
    return cu, cpp


def _inputs():
    cu, cpp = sources()
    hdr = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hdr += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return cu + cpp + hdr + [os.path.abspath(__file__)]


def _stamp_path():
    return os.path.join(BUILD, "machine.txt")


def up_to_date() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(_stamp_path()):
        return False
    with open(_stamp_path()) as f:
        if f.read().strip() != platform.machine():
            return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libpa.so; returns its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    cu, cpp = sources()
    jobs = []
    for src in cu:
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        jobs.append(([nvcc, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj], obj))
    for src in cpp:
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        jobs.append((["g++", *CXX_FLAGS, "-I" + _cuda_include(), "-c", src, "-o", obj], obj))
    logs = []
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for (cmd, _), out in zip(jobs, ex.map(lambda j: _run(j[0]), jobs)):
            logs.append("$ " + " ".join(cmd) + "\n" + out)
    tmp = LIB + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *[o for _, o in jobs], "-Xcompiler", "-fPIC"])
    os.replace(tmp, LIB)
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        f.write("\n".join(logs))
    with open(_stamp_path(), "w") as f:
        f.write(platform.machine())
    if verbose:
        print("\n".join(logs))
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
