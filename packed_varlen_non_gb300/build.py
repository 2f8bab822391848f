"""Builds the C-ABI library ``libh3attn.so`` in-tree for sm_103a.

Host C++ (plan builder, C-ABI layer) goes through g++, kernels through nvcc
with ``-gencode arch=compute_103a,code=sm_103a``; translation units compile in
parallel and link into one shared library under ``_build/`` next to this
file, with the CUDA runtime linked statically.  The plan builder is compiled
with ``-ffp-contract=off`` so that ``i*step + start`` is never fused.
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
LIB = os.path.join(OUT_DIR, "libh3attn.so")

CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

HOST_SOURCES = ["plan.cpp", "capi.cpp"]
CUDA_SOURCES = ["prologue.cu", "attn_fwd_tc.cu", "forward_noalloc.cu", "selftest.cu", "fp8_quant.cu"]
HEADERS = ["h3attn_internal.h", "device_common.cuh", "qk_norm.cuh"]

_ELF_MACHINE = {"x86_64": 62, "aarch64": 183, "arm64": 183}


def _deps():
    files = [os.path.join(CSRC, f) for f in HOST_SOURCES + CUDA_SOURCES + HEADERS]
    files += [os.path.join(INCLUDE, "h3attn.h"), os.path.abspath(__file__)]
    return files


def _lib_matches_host(path: str) -> bool:
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return False
    if len(head) < 20 or head[:4] != b"\x7fELF":
        return False
    machine = int.from_bytes(head[18:20], "little")
    return machine == _ELF_MACHINE.get(os.uname().machine, -1)


def is_stale() -> bool:
    if not os.path.exists(LIB) or not _lib_matches_host(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _deps())


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed:\n$ " + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compiles every translation unit and links libh3attn.so; returns its path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    cxx = shutil.which("g++") or "g++"
    common_inc = ["-I" + INCLUDE, "-I" + CSRC, "-I" + os.path.join(CUDA_HOME, "include")]
    jobs = []
    for src in HOST_SOURCES:
        obj = os.path.join(OUT_DIR, src + ".o")
        jobs.append([cxx, "-O2", "-std=c++17", "-fPIC", "-ffp-contract=off", "-Wall", *common_inc,
                     "-c", os.path.join(CSRC, src), "-o", obj])
    for src in CUDA_SOURCES:
        obj = os.path.join(OUT_DIR, src + ".o")
        cmd = [NVCC, *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
               "-Xcompiler", "-ffp-contract=off", *common_inc, "-c", os.path.join(CSRC, src),
               "-o", obj]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        jobs.append(cmd)
    logs = []
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        for out in ex.map(_run, jobs):
            logs.append(out)
    objs = [os.path.join(OUT_DIR, s + ".o") for s in HOST_SOURCES + CUDA_SOURCES]
    tmp = LIB + ".tmp"
    _run([NVCC, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    text = "".join(logs)
    if verbose and text.strip():
        print(text, file=sys.stderr)
    return text


def ensure_built() -> str:
    if is_stale():
        build()
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv))
    print(LIB)
