"""Builds ``libqa.so`` (the C ABI of include/qa.h) in-tree with nvcc for sm_103a.

Each .cu file compiles to an object in parallel; the objects link into one
shared library with the CUDA runtime linked statically, so the library loads
on a machine without a GPU (every CUDA call then fails with a status code).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libqa.so")
SOURCES = ["qa_api.cu", "k1_norm_rope_append.cu", "k2_prefill_tcgen05.cu", "k3_decode_splitkv.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
_lock = threading.Lock()


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqa.so")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "qa.h"))
    files.append(os.path.abspath(__file__))
    return files


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _compile(src: str, extra) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xptxas", "-v",
           "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC, *extra,
           "-c", os.path.join(CSRC, src), "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    with open(obj + ".log", "w") as fh:
        fh.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    return obj


def build(force: bool = False, extra=()) -> str:
    """Compile and link libqa.so if any source changed (or ``force``)."""
    with _lock:
        if not force and not stale():
            return LIB
        os.makedirs(BUILD, exist_ok=True)
        with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
            objs = list(ex.map(lambda s: _compile(s, list(extra)), SOURCES))
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static",
               "-Xlinker", "--version-script=" + os.path.join(CSRC, "libqa.map"), "-o", tmp, *objs]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
