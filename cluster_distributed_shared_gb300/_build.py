"""Builds libdsmemhist.so in-tree with nvcc for sm_103a (no torch extension
machinery, no cmake).  Translation units compile in parallel; the shared
library links the CUDA runtime statically."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libdsmemhist.so")

SOURCES = ["cluster_hist.cu", "cluster_ship.cu", "static_scratch.cu", "microbench.cu", "planner.cpp",
           "api.cpp"]
HEADERS = [os.path.join(CSRC, "internal.h"), os.path.join(CSRC, "ptx.cuh"),
           os.path.join(CSRC, "helper_split.h"), os.path.join(INCLUDE, "dsmem_hist.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-Wall,-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdsmemhist")
    return cand


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    objs, procs = [], []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(OUT_DIR, src + ".o")
        objs.append(obj)
        if force or _stale(obj, [path, *HEADERS]):
            cmd = [nvcc(), *ARCH, *COMMON, *extra_flags, "-c", path, "-o", obj]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT)))
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append(" ".join(cmd) + "\n" + text)
        elif verbose and text.strip():
            print(text, file=sys.stderr)
    if failed:
        raise RuntimeError("libdsmemhist build failed:\n" + "\n".join(failed))
    if force or procs or _stale(LIB_PATH, objs):
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            raise RuntimeError("libdsmemhist link failed:\n" + r.stdout.decode(errors="replace"))
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
