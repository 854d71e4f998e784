"""Python binding of libdsmemhist (the thread-block-cluster histogram).

Argument marshalling only: every step of the histogram runs in the CUDA
library (``csrc/``), called through its C ABI (``include/dsmem_hist.h``) with
ctypes.  PyTorch supplies device memory and the current stream.  There is no
CPU fallback: if the library is missing or the device cannot run it, the
calls raise.

Names follow the C ABI: ``dsmem_hist``, ``dsmem_hist_ex``,
``dsmem_hist_global_atomic``, ``dsmem_hist_host``, ``dsmem_hist_plan``,
``dsmem_hist_plan_ex``, ``dsmem_hist_plan_for_device``, ``dsmem_hist_release``.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsmemhist.so")

DSMEM_HIST_OK = 0
DSMEM_HIST_EINVAL = -1
DSMEM_HIST_EUNSUPPORTED = -2
DSMEM_HIST_ECUDA = -3
DSMEM_HIST_ETIMEOUT = -4
DSMEM_HIST_ENOMEM = -5

KERNEL_DIRECT = 0
KERNEL_SHIP = 1
SHIP_THREADS = 896  # DSMEM_HIST_SHIP_THREADS


class DsmemHistError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{message} [code {code}]")
        self.code = code


class Plan(ctypes.Structure):
    _fields_ = [
        ("cluster_size", ctypes.c_int32),
        ("bins_per_cta", ctypes.c_int32),
        ("passes", ctypes.c_int32),
        ("block_threads", ctypes.c_int32),
        ("num_clusters", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32),
        ("aggregate", ctypes.c_int32),
        ("ctas_per_sm", ctypes.c_int32),
        ("max_active_clusters", ctypes.c_int32),
        ("kernel", ctypes.c_int32),
        ("keys_per_thread", ctypes.c_int32),
        ("sub_vectors", ctypes.c_int32),
        ("hot_bin", ctypes.c_int32),
        ("partial_rows", ctypes.c_int32),
        ("partial_stride", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_int64),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class TuneResult(ctypes.Structure):
    _fields_ = [
        ("plan", Plan),
        ("global_atomic", ctypes.c_int32),
        ("ms", ctypes.c_float),
        ("control_ms", ctypes.c_float),
    ]


class MicrobenchResult(ctypes.Structure):
    _fields_ = [
        ("value", ctypes.c_double),
        ("ms", ctypes.c_double),
        ("bytes_per_s", ctypes.c_double),
        ("ops_expected", ctypes.c_uint64),
        ("ops_counted", ctypes.c_uint64),
        ("ctas", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class Request(ctypes.Structure):
    _fields_ = [
        ("cluster_size", ctypes.c_int32),
        ("block_threads", ctypes.c_int32),
        ("num_clusters", ctypes.c_int32),
        ("aggregate", ctypes.c_int32),
        ("max_slice_bytes", ctypes.c_int32),
        ("kernel", ctypes.c_int32),
        ("hot_bin_valid", ctypes.c_int32),
        ("hot_bin", ctypes.c_int32),
    ]


class Device(ctypes.Structure):
    _fields_ = [
        ("cc_major", ctypes.c_int32),
        ("cc_minor", ctypes.c_int32),
        ("sm_count", ctypes.c_int32),
        ("max_smem_per_block_optin", ctypes.c_int32),
        ("max_smem_per_sm", ctypes.c_int32),
        ("max_threads_per_sm", ctypes.c_int32),
        ("max_cluster_size", ctypes.c_int32),
    ]


EXPORTS = (
    "dsmem_hist", "dsmem_hist_ex", "dsmem_hist_global_atomic", "dsmem_hist_host",
    "dsmem_hist_partials", "dsmem_hist_reduce", "dsmem_hist_static", "dsmem_hist_tune",
    "dsmem_hist_microbench",
    "dsmem_hist_plan", "dsmem_hist_plan_ex", "dsmem_hist_plan_for_device", "dsmem_hist_strerror",
    "dsmem_hist_last_error", "dsmem_hist_release", "dsmem_hist_device_status",
    "dsmem_hist_version",
)

_lib = None
_lock = threading.Lock()


def lib():
    """The loaded libdsmemhist (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB_PATH)
            p, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            for name, args in [
                ("dsmem_hist", [p, i64, i32, p, p]),
                ("dsmem_hist_ex", [p, i64, i32, p, ctypes.POINTER(Request), p]),
                ("dsmem_hist_global_atomic", [p, i64, i32, p, p]),
                ("dsmem_hist_static", [p, i64, i32, p, p]),
                ("dsmem_hist_microbench", [i32, i32, i32, ctypes.POINTER(MicrobenchResult)]),
                ("dsmem_hist_tune", [p, i64, i32, i64, i32, ctypes.POINTER(TuneResult),
                                     ctypes.POINTER(i32), p]),
                ("dsmem_hist_host", [p, i64, i32, p, p]),
                ("dsmem_hist_partials", [p, i64, i32, ctypes.POINTER(Plan), p, i32, p]),
                ("dsmem_hist_reduce", [p, i32, i64, i32, p, p]),
                ("dsmem_hist_plan", [i32, i64, ctypes.POINTER(Plan)]),
                ("dsmem_hist_plan_ex", [i32, i64, ctypes.POINTER(Request), ctypes.POINTER(Plan)]),
                ("dsmem_hist_plan_for_device", [ctypes.POINTER(Device), i32, i64,
                                                ctypes.POINTER(Request), i32,
                                                ctypes.POINTER(Plan)]),
            ]:
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            L.dsmem_hist_strerror.argtypes = [ctypes.c_int]
            L.dsmem_hist_strerror.restype = ctypes.c_char_p
            L.dsmem_hist_last_error.argtypes = []
            L.dsmem_hist_last_error.restype = ctypes.c_char_p
            L.dsmem_hist_release.argtypes = []
            L.dsmem_hist_release.restype = None
            L.dsmem_hist_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
            L.dsmem_hist_device_status.restype = ctypes.c_int
            L.dsmem_hist_version.argtypes = []
            L.dsmem_hist_version.restype = ctypes.c_int
            _lib = L
    return _lib


def _check(code: int) -> None:
    if code != DSMEM_HIST_OK:
        L = lib()
        msg = L.dsmem_hist_last_error().decode(errors="replace") or \
            L.dsmem_hist_strerror(code).decode()
        raise DsmemHistError(code, msg)


def _request(cluster_size=0, block_threads=0, num_clusters=0, aggregate=-1, max_slice_bytes=0,
             kernel=-1, hot_bin=None):
    # hot_bin: None = automatic, a bin >= 0 = that hint, -1 = never the hot-bin kernel
    valid = 0 if hot_bin is None else (1 if hot_bin >= 0 else -1)
    return Request(cluster_size, block_threads, num_clusters, aggregate, max_slice_bytes, kernel,
                   valid, max(hot_bin or 0, 0))


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_keys(keys, num_bins):
    import torch
    if not isinstance(keys, torch.Tensor) or keys.dtype != torch.int32 or not keys.is_cuda:
        raise TypeError("keys must be a CUDA torch.int32 tensor")
    if not keys.is_contiguous():
        raise ValueError("keys must be contiguous")
    if not (1 <= int(num_bins) <= 2**31 - 1):
        raise ValueError("num_bins must be in [1, 2^31)")


def _out_bins(keys, num_bins, out):
    import torch
    if out is None:
        return torch.empty(int(num_bins), dtype=torch.int32, device=keys.device)
    if out.dtype not in (torch.int32, getattr(torch, "uint32", torch.int32)) or \
            out.numel() != num_bins or not out.is_contiguous() or out.device != keys.device:
        raise ValueError("out must be a contiguous 32-bit tensor of num_bins on the keys' device")
    return out


def dsmem_hist(keys, num_bins: int, out=None, stream=None, *, cluster_size=0, block_threads=0,
               num_clusters=0, aggregate=-1, max_slice_bytes=0, kernel=-1, hot_bin=None):
    """Histogram of a CUDA int32 tensor into `num_bins` 32-bit counters.

    Returns a torch.int32 tensor holding the uint32 counts bit for bit (use
    ``.view(torch.uint32)`` or numpy ``.view(np.uint32)`` to read them
    unsigned).  Asynchronous on `stream` (default: torch's current stream).
    Keyword arguments force parts of the launch shape (0 / -1 = planner);
    `hot_bin` names a bin expected to take a large share of the keys (None:
    automatic, from the previous histogram on the same stream; -1: never).
    """
    import torch
    _check_keys(keys, num_bins)
    out = _out_bins(keys, num_bins, out)
    with torch.cuda.device(keys.device):
        forced = (cluster_size, block_threads, num_clusters, max_slice_bytes) != (0, 0, 0, 0) \
            or aggregate != -1 or kernel != -1 or hot_bin is not None
        if forced:
            req = _request(cluster_size, block_threads, num_clusters, aggregate, max_slice_bytes,
                           kernel, hot_bin)
            _check(lib().dsmem_hist_ex(keys.data_ptr(), keys.numel(), int(num_bins),
                                       out.data_ptr(), ctypes.byref(req), _stream_handle(stream)))
        else:
            _check(lib().dsmem_hist(keys.data_ptr(), keys.numel(), int(num_bins), out.data_ptr(),
                                    _stream_handle(stream)))
    return out


def dsmem_hist_ex(keys, num_bins: int, request: Request, out=None, stream=None):
    """dsmem_hist with an explicit `Request` of planner overrides."""
    import torch
    _check_keys(keys, num_bins)
    out = _out_bins(keys, num_bins, out)
    with torch.cuda.device(keys.device):
        _check(lib().dsmem_hist_ex(keys.data_ptr(), keys.numel(), int(num_bins), out.data_ptr(),
                                   ctypes.byref(request), _stream_handle(stream)))
    return out


def dsmem_hist_static(keys, num_bins: int, out=None, stream=None):
    """dsmem_hist without any allocation by the library: the partial rows
    live in the library's fixed 32 MiB static device array (num_bins up to
    8,388,608).  For callers that cannot let a library allocate (stream
    capture, caller-owned memory arenas, allocator-free hot paths); calls
    that may overlap on the GPU share that array and must be serialised."""
    import torch
    _check_keys(keys, num_bins)
    out = _out_bins(keys, num_bins, out)
    with torch.cuda.device(keys.device):
        _check(lib().dsmem_hist_static(keys.data_ptr(), keys.numel(), int(num_bins),
                                       out.data_ptr(), _stream_handle(stream)))
    return out


def dsmem_hist_global_atomic(keys, num_bins: int, out=None, stream=None):
    """Comparison kernel: one global atomic per key (same result)."""
    import torch
    _check_keys(keys, num_bins)
    out = _out_bins(keys, num_bins, out)
    with torch.cuda.device(keys.device):
        _check(lib().dsmem_hist_global_atomic(keys.data_ptr(), keys.numel(), int(num_bins),
                                              out.data_ptr(), _stream_handle(stream)))
    return out


def dsmem_hist_host(keys, num_bins: int, out=None, stream=None):
    """Histogram of HOST keys (numpy int32 array or CPU torch.int32 tensor,
    ideally pinned) into host uint32 counts; synchronous.  Returns a numpy
    uint32 array, or fills `out` (numpy uint32 or CPU 32-bit tensor)."""
    import numpy as np
    import torch
    if isinstance(keys, torch.Tensor):
        if keys.is_cuda or keys.dtype != torch.int32 or not keys.is_contiguous():
            raise TypeError("keys must be a contiguous CPU torch.int32 tensor")
        kptr, n = keys.data_ptr(), keys.numel()
    else:
        if not isinstance(keys, np.ndarray) or keys.dtype != np.int32 or \
                not keys.flags.c_contiguous:
            raise TypeError("keys must be a contiguous numpy int32 array")
        kptr, n = keys.ctypes.data, keys.size
    if out is None:
        out = np.empty(int(num_bins), np.uint32)
    if isinstance(out, torch.Tensor):
        if out.is_cuda or out.numel() != num_bins or out.element_size() != 4:
            raise ValueError("out must be a CPU 32-bit tensor of num_bins")
        optr = out.data_ptr()
    else:
        if out.dtype != np.uint32 or out.size != num_bins or not out.flags.c_contiguous:
            raise ValueError("out must be a contiguous numpy uint32 array of num_bins")
        optr = out.ctypes.data
    if not (1 <= int(num_bins) <= 2**31 - 1):
        raise ValueError("num_bins must be in [1, 2^31)")
    _check(lib().dsmem_hist_host(kptr, n, int(num_bins), optr, _stream_handle(stream)))
    return out


def plan_struct(plan: dict) -> Plan:
    return Plan(**plan)


def dsmem_hist_partials(keys, num_bins: int, plan: dict, partials, accumulate: int = 0,
                        stream=None):
    """Stage 1: partial rows into caller-owned `partials` (a 16-byte aligned
    CUDA 32-bit tensor of workspace_bytes / 4 elements: partial_rows rows of
    partial_stride, then the helper's tile counter when the plan has a
    helper row); sum them with dsmem_hist_reduce(partials,
    plan["partial_rows"], ...)."""
    import torch
    _check_keys(keys, num_bins)
    need = -(-plan["workspace_bytes"] // 4)
    if not partials.is_cuda or partials.element_size() != 4 or partials.numel() < need or \
            not partials.is_contiguous():
        raise ValueError(f"partials must be a contiguous CUDA 32-bit tensor of >= {need}")
    ps = plan_struct(plan)
    with torch.cuda.device(keys.device):
        _check(lib().dsmem_hist_partials(keys.data_ptr(), keys.numel(), int(num_bins),
                                         ctypes.byref(ps), partials.data_ptr(), int(accumulate),
                                         _stream_handle(stream)))
    return partials


def dsmem_hist_reduce(partials, num_rows: int, partial_stride: int, num_bins: int, out=None,
                      stream=None):
    """Stage 2: sum the first `num_rows` partial rows (a plan's partial_rows)
    into `num_bins` counts."""
    import torch
    if not partials.is_cuda or partials.element_size() != 4 or \
            partials.numel() < num_rows * partial_stride:
        raise ValueError("partials too small")
    out = _out_bins(partials, num_bins, out)
    with torch.cuda.device(partials.device):
        _check(lib().dsmem_hist_reduce(partials.data_ptr(), int(num_rows), int(partial_stride),
                                       int(num_bins), out.data_ptr(), _stream_handle(stream)))
    return out


MICROBENCH_KINDS = {
    "local_red": 0,
    "remote_red": 1,
    "remote_st16_scattered": 2,
    "remote_st16_coalesced": 3,
    "cluster_barrier": 4,
    "dsmem_pingpong": 5,
    "gmem_pingpong": 6,
    "tile_exchange_dsmem": 7,
    "tile_exchange_gmem": 8,
}


def dsmem_hist_microbench(kind: str, cluster_size: int, iters: int = 4096) -> dict:
    """One DSMEM primitive on the current GPU (see the C header): ops (or
    bytes) per clock per SM, cycles per cluster barrier, cycles per one-way
    ping-pong hop, or milliseconds for the tile exchanges; with the work the
    probe issued (`ops_expected`) and counted on the device (`ops_counted`)."""
    r = MicrobenchResult()
    _check(lib().dsmem_hist_microbench(MICROBENCH_KINDS[kind], int(cluster_size), int(iters),
                                       ctypes.byref(r)))
    unit = {"cluster_barrier": "cycles/barrier", "remote_st16_scattered": "bytes/clk/SM",
            "remote_st16_coalesced": "bytes/clk/SM", "dsmem_pingpong": "cycles/hop",
            "gmem_pingpong": "cycles/hop", "tile_exchange_dsmem": "ms",
            "tile_exchange_gmem": "ms"}.get(kind, "ops/clk/SM")
    return {"kind": kind, "cluster_size": cluster_size, "iters": iters, "value": r.value,
            "unit": unit, "ms": r.ms, "bytes_per_s": r.bytes_per_s,
            "ops_expected": r.ops_expected, "ops_counted": r.ops_counted, "ctas": r.ctas}


def dsmem_hist_tune(keys, num_bins: int, sample_keys: int = 0, stream=None) -> list:
    """Times every legal cluster shape (and the global-atomics kernel) on a
    sample of `keys`; returns dicts sorted fastest first: plan fields plus
    `global_atomic`, `ms` and `control_ms`.  Synchronous."""
    import torch
    _check_keys(keys, num_bins)
    res = (TuneResult * 16)()
    count = ctypes.c_int32(0)
    with torch.cuda.device(keys.device):
        _check(lib().dsmem_hist_tune(keys.data_ptr(), keys.numel(), int(num_bins), int(sample_keys),
                                     16, res, ctypes.byref(count), _stream_handle(stream)))
    out = []
    for r in res[: count.value]:
        d = r.plan.as_dict()
        d.update(global_atomic=r.global_atomic, ms=r.ms, control_ms=r.control_ms)
        out.append(d)
    return out


def dsmem_hist_plan(num_bins: int, n: int, **overrides) -> dict:
    """The launch shape the library would use on the current device
    (``dsmem_hist_plan``; with keyword overrides, ``dsmem_hist_plan_ex``)."""
    plan = Plan()
    if overrides:
        req = _request(**overrides)
        _check(lib().dsmem_hist_plan_ex(int(num_bins), int(n), ctypes.byref(req),
                                        ctypes.byref(plan)))
    else:
        _check(lib().dsmem_hist_plan(int(num_bins), int(n), ctypes.byref(plan)))
    return plan.as_dict()


def dsmem_hist_plan_ex(num_bins: int, n: int, request: Request) -> dict:
    """dsmem_hist_plan with an explicit `Request` of planner overrides."""
    plan = Plan()
    _check(lib().dsmem_hist_plan_ex(int(num_bins), int(n), ctypes.byref(request),
                                    ctypes.byref(plan)))
    return plan.as_dict()


def dsmem_hist_plan_for_device(device: dict, num_bins: int, n: int, max_active_clusters: int = 0,
                               **overrides) -> dict:
    """Plan for a described device (host logic only; no CUDA call)."""
    dev = Device(**device)
    plan = Plan()
    req = _request(**overrides)
    _check(lib().dsmem_hist_plan_for_device(ctypes.byref(dev), int(num_bins), int(n),
                                            ctypes.byref(req), int(max_active_clusters),
                                            ctypes.byref(plan)))
    return plan.as_dict()


def dsmem_hist_release() -> None:
    lib().dsmem_hist_release()


def dsmem_hist_device_status() -> int:
    """Reads and clears the ship kernel's device status word (0: every
    bounded inbox wait succeeded since the last call)."""
    word = ctypes.c_uint32(0)
    rc = lib().dsmem_hist_device_status(ctypes.byref(word))
    if rc not in (DSMEM_HIST_OK, DSMEM_HIST_ETIMEOUT):
        _check(rc)
    return word.value


def dsmem_hist_version() -> int:
    return lib().dsmem_hist_version()


def strerror(code: int) -> str:
    return lib().dsmem_hist_strerror(code).decode()
