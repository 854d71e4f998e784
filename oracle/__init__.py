"""CPU oracle for the cluster histogram -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library never calls it and has no
CPU fallback.

``histogram(keys, num_bins)`` runs the single-threaded C loop in
``oracle.c`` (compiled with gcc into ``liboracle.so`` on first use): the plain
count of each bin in [0, num_bins), keys outside that range ignored, 32-bit
counters ("Distributed Shared Memory", section "The cluster histogram").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
import time

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain -O2, portable)."""
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
        ):
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC])
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_histogram.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                         ctypes.c_void_p]
        lib.oracle_histogram.restype = None
        _lib = lib
    return _lib


def histogram(keys: np.ndarray, num_bins: int, out: np.ndarray | None = None) -> np.ndarray:
    """uint32[num_bins]: count of each bin b in [0, num_bins) among `keys`."""
    keys = np.ascontiguousarray(keys, dtype=np.int32)
    if not (1 <= num_bins <= 2**31 - 1):
        raise ValueError("num_bins must be in [1, 2^31)")
    out = np.empty(num_bins, np.uint32) if out is None else out
    assert out.dtype == np.uint32 and out.size == num_bins and out.flags.c_contiguous
    _load().oracle_histogram(keys.ctypes.data, keys.size, num_bins, out.ctypes.data)
    return out


def time_histogram(keys: np.ndarray, num_bins: int, min_seconds: float = 10.0,
                   max_reps: int = 50):
    """Time the oracle as it stands on this host (one thread).

    Repeats the full call until `min_seconds` of CPU work have run (at least
    once).  Returns (median seconds per call, repetitions).
    """
    out = np.empty(num_bins, np.uint32)
    times = []
    t_total = 0.0
    while not times or (t_total < min_seconds and len(times) < max_reps):
        t0 = time.perf_counter()
        histogram(keys, num_bins, out)
        dt = time.perf_counter() - t0
        times.append(dt)
        t_total += dt
    times.sort()
    return times[len(times) // 2], len(times)
