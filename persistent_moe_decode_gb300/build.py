"""Builds the C-ABI library libmk.so in-tree (sm_103a only, no cmake).

    python -m persistent_moe_decode_gb300.build [--force]

The kernel translation unit is compiled by nvcc for sm_103a; the host
scheduler and ABI by the host compiler; the three objects are linked against
the shared CUDA runtime.  Objects go to ``_build/`` next to the package.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmk.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home() -> str:
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.exists(os.path.join(c, "bin", "nvcc")):
            return c
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(nvcc))
    raise RuntimeError("nvcc not found: set CUDA_HOME")


def _sources():
    return [os.path.join(CSRC, f) for f in ("mk_kernel.cu", "mk_static.cu", "mk_service.cu", "mk_sched.cpp",
                                             "mk_api.cpp")]


def _deps():
    return _sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))] + \
        [os.path.join(INCLUDE, "mk.h")]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    os.makedirs(BUILD, exist_ok=True)
    cxx = shutil.which("g++") or "c++"
    common_inc = [f"-I{INCLUDE}", f"-I{CSRC}", f"-I{os.path.join(cuda, 'include')}"]
    jobs = []
    for src in _sources():
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        if src.endswith(".cu"):
            cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-Xptxas", "-v" if verbose else "-O3", *common_inc, "-c", src, "-o", obj]
        else:
            cmd = [cxx, "-O2", "-std=c++17", "-fPIC", "-Wall", *common_inc, "-c", src, "-o", obj]
        jobs.append((cmd, obj))

    def run(job):
        cmd, obj = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stderr

    with ThreadPoolExecutor(len(jobs)) as ex:
        logs = list(ex.map(run, jobs))
    if verbose:
        for lg in logs:
            if lg:
                sys.stderr.write(lg)
    tmp = LIB + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *[o for _, o in jobs],
            f"-L{os.path.join(cuda, 'lib64')}", "-Xlinker", f"-rpath={os.path.join(cuda, 'lib64')}"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(link)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
