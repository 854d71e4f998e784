"""Seeded synthetic key generators (inputs only; no histogram arithmetic).

Both sides of every parity check -- the CPU oracle and the CUDA library --
receive keys produced here.  The C source (``gen.c``) is compiled with gcc on
first use into ``libgen.so`` next to it.  Generation is split across host
threads: the SplitMix64 counter form makes every index range independent, so
the bytes do not depend on the thread count.

Workloads are named by what they are.  The five synthetic workloads of the
cluster-histogram study:

=====================  =============  ========  =======================================
name                   keys           bins      distribution
=====================  =============  ========  =======================================
uniform-1M-8K          1,048,576      8,192     uniform on [0, 8192)
uniform-64M-64K        67,108,864     65,536    uniform on [0, 65536)
uniform-256M-256K      268,435,456    262,144   uniform on [0, 262144)
zipf1.1-256M-256K      268,435,456    262,144   Zipf(s=1.1) ranks, randomly permuted
runs256-1G-512K        1,073,741,824  524,288   50% uniform, 50% runs of 256 equal keys
=====================  =============  ========  =======================================

and one skewed case beside them: hot25-256M-256K, 268,435,456 keys over 262,144
bins, of which a quarter (each key independently with probability 1/4) are one
hot bin drawn from the seed and the rest uniform.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "libgen.so")
_lock = threading.Lock()
_lib = None

WORKLOADS = {
    "uniform-1M-8K": dict(n=1 << 20, num_bins=8192, dist="uniform"),
    "uniform-64M-64K": dict(n=1 << 26, num_bins=65536, dist="uniform"),
    "uniform-256M-256K": dict(n=1 << 28, num_bins=262144, dist="uniform"),
    "zipf1.1-256M-256K": dict(n=1 << 28, num_bins=262144, dist="zipf", s=1.1),
    "runs256-1G-512K": dict(n=1 << 30, num_bins=524288, dist="runs", run_len=256),
    "hot25-256M-256K": dict(n=1 << 28, num_bins=262144, dist="hot", share=0.25),
}


def build(force: bool = False) -> str:
    """Compile gen.c into libgen.so (gcc, portable flags only)."""
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
        ):
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.check_call(
                ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
            )
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, u32, u64 = ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64
        p = ctypes.c_void_p
        lib.gen_splitmix64_draw.argtypes = [u64, u64]
        lib.gen_splitmix64_draw.restype = u64
        lib.gen_uniform.argtypes = [p, i64, i64, u32, u64]
        lib.gen_uniform.restype = None
        lib.gen_runs.argtypes = [p, i64, i64, i64, u32, u32, u64]
        lib.gen_runs.restype = None
        lib.gen_zipf.argtypes = [p, i64, i64, u32, ctypes.c_double, u64]
        lib.gen_zipf.restype = ctypes.c_int
        lib.gen_zipf_tables.argtypes = [u32, ctypes.c_double, u64, p, p]
        lib.gen_zipf_tables.restype = ctypes.c_int
        lib.gen_hot.argtypes = [p, i64, i64, u32, u32, u64]
        lib.gen_hot.restype = None
        lib.gen_hot_bin.argtypes = [u32, u64]
        lib.gen_hot_bin.restype = u32
        _lib = lib
    return _lib


def splitmix64(seed: int, i: int) -> int:
    """Draw number i of the SplitMix64 stream with this seed."""
    return int(_load().gen_splitmix64_draw(seed & (2**64 - 1), i))


def _fill(out: np.ndarray, fn, threads: int | None) -> np.ndarray:
    n = out.size
    threads = threads or min(32, os.cpu_count() or 1)
    chunk = max(1 << 20, -(-n // threads))
    spans = [(o, min(chunk, n - o)) for o in range(0, n, chunk)]
    base = out.ctypes.data

    def run(span):
        off, cnt = span
        fn(ctypes.c_void_p(base + 4 * off), off, cnt)

    if len(spans) <= 1:
        for s in spans:
            run(s)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(run, spans))
    return out


def uniform(n: int, num_bins: int, seed: int, out: np.ndarray | None = None,
            threads: int | None = None) -> np.ndarray:
    """Keys uniform on [0, num_bins) (exact for power-of-two num_bins)."""
    lib = _load()
    out = np.empty(n, np.int32) if out is None else out
    return _fill(out, lambda p, o, c: lib.gen_uniform(p, o, c, num_bins, seed), threads)


def runs(n: int, num_bins: int, seed: int, run_len: int = 256,
         out: np.ndarray | None = None, threads: int | None = None) -> np.ndarray:
    """First n//2 keys uniform; the rest in runs of run_len equal keys."""
    lib = _load()
    out = np.empty(n, np.int32) if out is None else out
    return _fill(out, lambda p, o, c: lib.gen_runs(p, o, c, n, num_bins, run_len, seed),
                 threads)


def zipf(n: int, num_bins: int, seed: int, s: float = 1.1,
         out: np.ndarray | None = None, threads: int | None = None) -> np.ndarray:
    """Truncated Zipf(s) over ranks 1..num_bins, ranks permuted to bin ids."""
    lib = _load()
    out = np.empty(n, np.int32) if out is None else out

    def fn(p, o, c):
        if lib.gen_zipf(p, o, c, num_bins, s, seed) != 0:
            raise MemoryError("gen_zipf: table allocation failed")

    return _fill(out, fn, threads)


def hot_bin(num_bins: int, seed: int) -> int:
    """The hot bin of `hot` for this seed."""
    return int(_load().gen_hot_bin(num_bins, seed & (2**64 - 1)))


def hot(n: int, num_bins: int, seed: int, share: float = 0.25, out: np.ndarray | None = None,
        threads: int | None = None) -> np.ndarray:
    """Each key is hot_bin(num_bins, seed) with probability `share`, else
    uniform on [0, num_bins)."""
    lib = _load()
    out = np.empty(n, np.int32) if out is None else out
    thr = min(int(round(share * 2**32)), 2**32 - 1)
    return _fill(out, lambda p, o, c: lib.gen_hot(p, o, c, num_bins, thr, seed), threads)


def zipf_tables(num_bins: int, s: float, seed: int):
    """(cdf over ranks, rank -> bin permutation) exactly as gen_zipf uses them."""
    cdf = np.empty(num_bins, np.float64)
    perm = np.empty(num_bins, np.uint32)
    if _load().gen_zipf_tables(num_bins, s, seed, cdf.ctypes.data, perm.ctypes.data) != 0:
        raise MemoryError("gen_zipf_tables failed")
    return cdf, perm


def workload(name: str, seed: int, out: np.ndarray | None = None,
             threads: int | None = None, n: int | None = None) -> np.ndarray:
    """Keys of one named workload (see the module table) for this seed; `n`
    scales it to another length with the same distribution and layout."""
    w = WORKLOADS[name]
    n = w["n"] if n is None else n
    if w["dist"] == "uniform":
        return uniform(n, w["num_bins"], seed, out, threads)
    if w["dist"] == "zipf":
        return zipf(n, w["num_bins"], seed, w["s"], out, threads)
    if w["dist"] == "runs":
        return runs(n, w["num_bins"], seed, w["run_len"], out, threads)
    if w["dist"] == "hot":
        return hot(n, w["num_bins"], seed, w["share"], out, threads)
    raise KeyError(name)
