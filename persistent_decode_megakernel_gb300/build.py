"""Builds the C-ABI library libmbk.so in-tree (nvcc for sm_103a, g++ for the host scheduler).

Translation units compile in parallel into persistent_decode_megakernel_gb300/_build/ and link
into persistent_decode_megakernel_gb300/libmbk.so.  Rebuilds only when a source is newer than the
library.  Usage: python -m persistent_decode_megakernel_gb300.build [--force]
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmbk.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"

CU_SOURCES = ["mbk_kernel.cu", "mbk_api.cu", "mbk_static.cu", "mbk_prefill.cu"]
CPP_SOURCES = ["mbk_sched.cpp", "mbk_simulate.cpp", "mbk_args.cpp"]
HEADERS = ["mbk_plan.h", "mbk_device.h", "mbk_sched.h", "mbk_prefill.h", "mbk_args.h"]


def _cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or "/usr/local/cuda"
    if not os.path.exists(os.path.join(home, "bin", "nvcc")):
        nvcc = shutil.which("nvcc")
        if nvcc:
            home = os.path.dirname(os.path.dirname(nvcc))
    return home


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in CU_SOURCES + CPP_SOURCES + HEADERS]
    paths.append(os.path.join(INCLUDE, "mbk.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build step failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libmbk.so if needed; returns its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    os.makedirs(OUT_DIR, exist_ok=True)
    jobs = []
    for f in CU_SOURCES:
        obj = os.path.join(OUT_DIR, f + ".o")
        jobs.append([nvcc, ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xptxas", "-v", "-Xcompiler", "-fPIC",
                     "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, f), "-o", obj])
    for f in CPP_SOURCES:
        obj = os.path.join(OUT_DIR, f + ".o")
        jobs.append(["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-I", INCLUDE, "-I", CSRC,
                     "-c", os.path.join(CSRC, f), "-o", obj])
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        logs = list(ex.map(_run, jobs))
    if verbose:
        for lg in logs:
            sys.stdout.write(lg)
    objs = [os.path.join(OUT_DIR, f + ".o") for f in CU_SOURCES + CPP_SOURCES]
    tmp = LIB + f".tmp{os.getpid()}"
    _run([nvcc, ARCH, "-shared", "-o", tmp] + objs +
         ["-cudart", "shared", "-Xlinker", "-rpath", "-Xlinker", os.path.join(cuda, "lib64")])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
