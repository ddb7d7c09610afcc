"""Build libpa.so (the C-ABI library) in-tree for sm_103a.

Each translation unit is compiled in parallel with nvcc
(``-gencode arch=compute_103a,code=sm_103a -lineinfo -O3``), then linked
into ``paged_kv_cache_35_gb300/libpa.so`` with the CUDA runtime linked
statically.  Nothing is installed anywhere else.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(HERE, "libpa.so")

CU_SOURCES = ["pa_cache_ops.cu", "pa_decode.cu", "pa_prefill.cu", "pa_graph.cu", "pa_checks.cu"]
CPP_SOURCES = ["pa_allocator.cpp"]
HEADERS = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] + [
    os.path.join(ROOT, "include", "pa.h")
]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
                     "-Xptxas", "-warn-spills"]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest(paths) -> float:
    return max(os.path.getmtime(p) for p in paths if os.path.exists(p))


def _up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    srcs = [os.path.join(CSRC, f) for f in CU_SOURCES + CPP_SOURCES] + HEADERS + [__file__]
    return os.path.getmtime(LIB_PATH) >= _newest(srcs)


def build(force: bool = False, verbose: bool = False, extra_nvcc=()) -> str:
    if not force and _up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    objs = []
    for f in CU_SOURCES:
        obj = os.path.join(BUILD_DIR, f + ".o")
        cmd = [nvcc, *NVCC_FLAGS, *extra_nvcc, "-c", os.path.join(CSRC, f), "-o", obj]
        jobs.append((f, cmd))
        objs.append(obj)
    for f in CPP_SOURCES:
        obj = os.path.join(BUILD_DIR, f + ".o")
        cmd = ["g++", *CXX_FLAGS, "-c", os.path.join(CSRC, f), "-o", obj]
        jobs.append((f, cmd))
        objs.append(obj)
    procs = [(f, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True))
             for f, cmd in jobs]
    failed = []
    for f, cmd, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            sys.stderr.write(f"[build] {' '.join(cmd)}\n{out}")
        if p.returncode != 0:
            failed.append(f)
    if failed:
        raise RuntimeError(f"compilation failed: {failed}")
    tmp = LIB_PATH + ".tmp"
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lstdc++"]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB_PATH)
