"""The C ABI without a GPU: the library loads, exports every declared entry
point, rejects bad arguments before touching CUDA, and plans shapes for a
described device (host logic only)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import cluster_distributed_shared_gb300 as pkg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

GB300 = dict(cc_major=10, cc_minor=3, sm_count=152, max_smem_per_block_optin=232448,
             max_smem_per_sm=233472, max_threads_per_sm=2048, max_cluster_size=16)
H100 = dict(cc_major=9, cc_minor=0, sm_count=132, max_smem_per_block_optin=232448,
            max_smem_per_sm=233472, max_threads_per_sm=2048, max_cluster_size=16)


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"^DSMEM_HIST_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, re.M)
    return names


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert "dsmem_hist" in names and len(names) >= 10
    L = pkg.lib()
    for name in names:
        assert hasattr(L, name), name
    assert set(pkg.EXPORTS) <= set(names)


def test_header_compiles_as_c_and_links(tmp_path):
    # A C11 program (tests/c_abi_check.c) includes the header and calls the
    # host-only entry points through libdsmemhist.so: the boundary is a C ABI.
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    from cluster_distributed_shared_gb300 import _build
    lib = pkg.lib()._name
    cuda_inc = None
    for base in filter(None, [os.environ.get("CUDA_HOME"), os.path.dirname(os.path.dirname(_build.nvcc())),
                              "/usr/local/cuda"]):
        if os.path.exists(os.path.join(base, "include", "cuda_runtime_api.h")):
            cuda_inc = os.path.join(base, "include")
            break
    if cuda_inc is None:
        pytest.skip("cuda_runtime_api.h not found")
    exe = str(tmp_path / "c_abi_check")
    cmd = [gcc, "-std=c11", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
           os.path.join(ROOT, "tests", "c_abi_check.c"), lib,
           "-Wl,-rpath," + os.path.dirname(lib), "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip().endswith("ok")
    assert f"block_threads={pkg.SHIP_THREADS}" in out.stdout


def test_helper_split_controller(tmp_path):
    # tests/helper_split_check.cpp drives the idle-SM helper's share
    # controller and tile split (csrc/helper_split.h, the code the library's
    # launcher runs) with synthetic reports: prior, convergence without
    # overshoot, clamps, ignored targets, damping on direction changes, the
    # stale-report window (with wrap-around), whole-round splits.
    import shutil
    import subprocess
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no g++")
    exe = str(tmp_path / "helper_split_check")
    cmd = [gxx, "-std=c++17", "-O2", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "cluster_distributed_shared_gb300", "csrc"),
           os.path.join(ROOT, "tests", "helper_split_check.cpp"), "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip() == "ok"


def test_version_and_strerror():
    assert pkg.dsmem_hist_version() >= 100
    for code in (0, -1, -2, -3, -4, -5):
        assert pkg.strerror(code).startswith("DSMEM_HIST")


@pytest.mark.parametrize("fn", ["dsmem_hist", "dsmem_hist_global_atomic", "dsmem_hist_host"])
def test_invalid_arguments_rejected_before_cuda(fn):
    L = pkg.lib()
    f = getattr(L, fn)
    buf = (ctypes.c_uint32 * 8)()
    p = ctypes.cast(buf, ctypes.c_void_p)
    cases = [
        (p, -1, 8, p),              # n < 0
        (p, 4, 0, p),               # num_bins < 1
        (p, 4, -5, p),              # num_bins < 1
        (None, 4, 8, p),            # keys NULL with n > 0
        (p, 4, 8, None),            # bins NULL
        (ctypes.c_void_p(ctypes.addressof(buf) + 2), 1, 8, p),  # misaligned keys
        (p, 1, 8, ctypes.c_void_p(ctypes.addressof(buf) + 1)),  # misaligned bins
    ]
    for keys, n, nb, bins in cases:
        assert f(keys, n, nb, bins, None) == pkg.DSMEM_HIST_EINVAL
        assert L.dsmem_hist_last_error()


def plan(dev, nb, n, mac=0, **kw):
    return pkg.dsmem_hist_plan_for_device(dev, nb, n, mac, **kw)


@pytest.mark.parametrize("nb,n,P,S", [
    (8192, 1 << 20, 2, 4096),
    (65536, 1 << 26, 2, 32768),
    (262144, 1 << 28, 8, 32768),
    (524288, 1 << 30, 16, 32768),
])
def test_planner_matches_published_cluster_shapes(nb, n, P, S):
    p = plan(GB300, nb, n, cluster_size=P)
    assert (p["cluster_size"], p["bins_per_cta"], p["passes"]) == (P, S, 1)
    assert p["kernel"] == pkg.KERNEL_SHIP and p["block_threads"] == pkg.SHIP_THREADS
    assert 4 * S < p["smem_bytes"] <= GB300["max_smem_per_block_optin"]
    q = plan(GB300, nb, n)          # the planner's own choice agrees here
    assert (q["cluster_size"], q["bins_per_cta"]) == (P, S)
    d = plan(GB300, nb, n, cluster_size=P, kernel=pkg.KERNEL_DIRECT)
    assert d["kernel"] == pkg.KERNEL_DIRECT and d["smem_bytes"] == 4 * S


@pytest.mark.parametrize("nb", [1, 2, 3, 5, 97, 4095, 4096, 4097, 65535, 65537, 100003, 262143,
                                524289, 929792, 929793, 1 << 22, 2**31 - 1])
@pytest.mark.parametrize("slice_cap", [0, 1024, 232448])
def test_planner_covers_every_bin(nb, slice_cap):
    for forced in (0, 1, 2, 16):
        p = plan(GB300, nb, 1 << 20, cluster_size=forced, max_slice_bytes=slice_cap)
        P, S, passes = p["cluster_size"], p["bins_per_cta"], p["passes"]
        assert S % 4 == 0 and S >= 4
        cap = (slice_cap or 128 * 1024)
        assert 4 * S <= min(cap, GB300["max_smem_per_block_optin"]) or 4 * S == 16
        assert passes * P * S >= nb                       # no bin dropped
        assert (passes - 1) * P * S < nb                  # no empty pass
        assert P * S < 2 ** 20 + 16 * 4                    # owner arithmetic range
        assert p["partial_stride"] % 4 == 0 and p["partial_stride"] >= nb
        helper = p["partial_rows"] - p["num_clusters"]
        assert helper in (0, 1)                            # the helper's row, if any
        assert not helper or (p["kernel"] == pkg.KERNEL_SHIP and passes == 1)
        assert p["workspace_bytes"] == p["partial_rows"] * p["partial_stride"] * 4 + 32 * helper
        assert p["smem_bytes"] <= GB300["max_smem_per_block_optin"]
        if p["kernel"] == pkg.KERNEL_SHIP:
            assert P >= 2 and p["block_threads"] == pkg.SHIP_THREADS
            assert p["keys_per_thread"] in (4, 8)
            nq = p["sub_vectors"]   # staging rows per owner block
            assert nq >= 1 and nq * 32 * P >= 1.5 * pkg.SHIP_THREADS * p["keys_per_thread"]
            assert p["smem_bytes"] == 4 * S + ship_staging(P, nq)
            assert S < 0xFFFF                               # 16-bit local indices + sentinel
        else:
            assert p["smem_bytes"] == 4 * S
        if forced:
            assert P == forced


def ship_staging(P, rows):
    # padding counters, three cursor sets of P + 1 rows, headers + sink +
    # mbarriers, two staging and two inbox buffers of P blocks of `rows`
    # rows of 64 bytes
    return 4 * 32 + 3 * 4 * 32 * (P + 1) + 256 + 4 * P * rows * 64


@pytest.mark.parametrize("P", range(2, 17))
def test_ship_plan_fits_for_every_cluster_size(P):
    for nb in (P * 4, P * 32768, 262144, 524288):
        p = plan(GB300, nb, 1 << 26, cluster_size=P, kernel=pkg.KERNEL_SHIP)
        assert p["kernel"] == pkg.KERNEL_SHIP
        assert p["smem_bytes"] + 1024 <= GB300["max_smem_per_sm"]
        # staging columns hold at least 1.5 times the expected keys per (owner, lane) and round
        expected = pkg.SHIP_THREADS // 32 * p["keys_per_thread"] / P
        assert p["sub_vectors"] >= 1.5 * expected


def test_owner_magic_exact():
    # owner = (rel * (floor(2^40 / S) + 1)) >> 40 must equal rel // S for every
    # rel < P * S the kernel can see (checked exhaustively at the slice sizes'
    # extremes, and on a grid in between).
    for S in [4, 8, 12, 4096, 25004, 32768, 58108, 58112]:
        magic = (1 << 40) // S + 1
        P = 16
        rels = list(range(0, min(P * S, 200000))) + list(range(max(0, P * S - 200000), P * S))
        for rel in rels[:: max(1, len(rels) // 50000)] + [P * S - 1, P * S]:
            assert (rel * magic) >> 40 == rel // S, (S, rel)   # P * S: the clamp value


def test_planner_grid_and_threads():
    p = plan(GB300, 262144, 1 << 28, mac=16)
    assert p["num_clusters"] == 16 and p["block_threads"] == pkg.SHIP_THREADS
    assert p["ctas_per_sm"] == 1
    small = plan(GB300, 8192, 1000, mac=100)
    assert small["num_clusters"] == 1 and small["block_threads"] == pkg.SHIP_THREADS
    direct = plan(GB300, 8192, 1000, mac=100, kernel=pkg.KERNEL_DIRECT)
    assert direct["block_threads"] == 512 and direct["kernel"] == pkg.KERNEL_DIRECT
    one = plan(GB300, 8192, 1 << 20, cluster_size=1)
    assert one["kernel"] == pkg.KERNEL_DIRECT      # no remote owners: local increments
    # Ship kernel: about two rounds (896 threads x 8 keys) per CTA; direct
    # kernel: four unrolled steps (16 keys per thread) per CTA.
    ship = plan(GB300, 8192, 1 << 20, mac=76)
    assert ship["kernel"] == pkg.KERNEL_SHIP and ship["keys_per_thread"] == 8
    assert ship["num_clusters"] == -(-(1 << 20) // (2 * pkg.SHIP_THREADS * 8 * 2)) == 37
    assert plan(GB300, 8192, 1 << 30, mac=76)["num_clusters"] == 76
    d = plan(GB300, 8192, 1 << 20, mac=76, kernel=pkg.KERNEL_DIRECT)
    assert d["num_clusters"] == -(-(1 << 20) // (2 * d["block_threads"] * 16 * 4))
    forced = plan(GB300, 8192, 1 << 20, mac=100, num_clusters=7, block_threads=256)
    assert forced["num_clusters"] == 7 and forced["block_threads"] == 256


def test_planner_keeps_huge_inputs_off_the_ship_kernel():
    # The ship kernel indexes warp tiles with 32-bit integers: from 2^38 keys
    # on the planner picks the direct kernel, and refuses a forced ship kernel.
    assert plan(GB300, 262144, (1 << 38) - 1, mac=15)["kernel"] == pkg.KERNEL_SHIP
    big = plan(GB300, 262144, 1 << 38, mac=15)
    assert big["kernel"] == pkg.KERNEL_DIRECT and big["cluster_size"] == 8
    with pytest.raises(pkg.DsmemHistError) as e:
        plan(GB300, 262144, 1 << 38, mac=15, kernel=pkg.KERNEL_SHIP)
    assert e.value.code == pkg.DSMEM_HIST_EINVAL


def test_planner_multi_pass_when_bins_exceed_cluster():
    p = plan(GB300, 1 << 22, 1 << 24)
    assert p["cluster_size"] == 16 and p["passes"] == 8 and p["bins_per_cta"] == 32768
    p8 = dict(GB300, max_cluster_size=8)
    q = plan(p8, 524288, 1 << 24)
    assert q["cluster_size"] == 8 and q["passes"] == 2


def test_planner_errors():
    old = dict(H100, cc_major=8)
    with pytest.raises(pkg.DsmemHistError) as e:
        plan(old, 1024, 10)
    assert e.value.code == pkg.DSMEM_HIST_EUNSUPPORTED
    with pytest.raises(pkg.DsmemHistError) as e:
        plan(dict(GB300, max_cluster_size=8), 1024, 10, cluster_size=16)
    assert e.value.code == pkg.DSMEM_HIST_EUNSUPPORTED
    for bad in [dict(cluster_size=17), dict(block_threads=100), dict(block_threads=2048),
                dict(num_clusters=-1)]:
        with pytest.raises(pkg.DsmemHistError) as e:
            plan(GB300, 1024, 10, **bad)
        assert e.value.code == pkg.DSMEM_HIST_EINVAL
    with pytest.raises(pkg.DsmemHistError):
        plan(GB300, 0, 10)


def test_aggregate_and_kernel_overrides():
    d = pkg.KERNEL_DIRECT
    assert plan(GB300, 4096, 1 << 20, aggregate=0, kernel=d)["aggregate"] == 0
    assert plan(GB300, 4096, 1 << 20, aggregate=1, kernel=d)["aggregate"] == 1
    assert plan(GB300, 4096, 1 << 20, kernel=d)["aggregate"] == 0
    assert plan(GB300, 4096, 1 << 20)["kernel"] == pkg.KERNEL_SHIP
    assert plan(GB300, 4096, 1 << 20, block_threads=256)["kernel"] == d
    for bad in [dict(kernel=pkg.KERNEL_SHIP, cluster_size=1),
                dict(kernel=pkg.KERNEL_SHIP, block_threads=256), dict(kernel=7)]:
        with pytest.raises(pkg.DsmemHistError) as e:
            plan(GB300, 4096, 1 << 20, **bad)
        assert e.value.code == pkg.DSMEM_HIST_EINVAL


def test_tune_and_microbench_reject_bad_arguments():
    L = pkg.lib()
    buf = (ctypes.c_uint32 * 8)()
    p = ctypes.cast(buf, ctypes.c_void_p)
    count = ctypes.c_int32(0)
    res = (pkg.TuneResult * 2)()
    assert L.dsmem_hist_tune(p, -1, 8, 0, 2, res, ctypes.byref(count), None) == pkg.DSMEM_HIST_EINVAL
    assert L.dsmem_hist_tune(p, 4, 0, 0, 2, res, ctypes.byref(count), None) == pkg.DSMEM_HIST_EINVAL
    r = ctypes.byref(pkg.MicrobenchResult())
    assert L.dsmem_hist_microbench(0, 17, 16, r) == pkg.DSMEM_HIST_EINVAL
    assert L.dsmem_hist_microbench(0, 2, 0, r) == pkg.DSMEM_HIST_EINVAL
    assert L.dsmem_hist_microbench(0, 2, 16, None) == pkg.DSMEM_HIST_EINVAL
    # ping-pong needs two CTAs and a bounded number of rounds
    assert L.dsmem_hist_microbench(5, 1, 16, r) == pkg.DSMEM_HIST_EINVAL
    assert L.dsmem_hist_microbench(6, 2, (1 << 20) + 1, r) == pkg.DSMEM_HIST_EINVAL
    # the tile exchange pairs CTAs 2j and 2j + 1: an even cluster size
    assert L.dsmem_hist_microbench(7, 3, 16, r) == pkg.DSMEM_HIST_EINVAL
    assert L.dsmem_hist_microbench(8, 1, 16, r) == pkg.DSMEM_HIST_EINVAL
    assert L.dsmem_hist_microbench(9, 2, 16, r) == pkg.DSMEM_HIST_EINVAL


def test_ship_threads_match_header():
    header = open(os.path.join(ROOT, "include", "dsmem_hist.h")).read()
    m = re.search(r"^#define DSMEM_HIST_SHIP_THREADS (\d+)", header, re.M)
    assert m and int(m.group(1)) == pkg.SHIP_THREADS
    assert pkg.SHIP_THREADS % 32 == 0 and 32 * 17 <= pkg.SHIP_THREADS <= 1024


def test_planner_hot_bin_hint():
    p = plan(GB300, 262144, 1 << 28, 15)
    assert p["hot_bin"] == -1                      # no hint: the default kernel
    h = plan(GB300, 262144, 1 << 28, 15, hot_bin=146157)
    assert h["hot_bin"] == 146157 and h["kernel"] == pkg.KERNEL_SHIP
    skip = ("hot_bin", "partial_rows", "workspace_bytes")
    assert {k: v for k, v in h.items() if k not in skip} == \
        {k: v for k, v in p.items() if k not in skip}   # same shape otherwise
    assert h["partial_rows"] == p["partial_rows"]           # the helper runs with either kernel
    assert plan(GB300, 262144, 1 << 28, 15, hot_bin=0)["hot_bin"] == 0
    # the direct kernel ignores the hint
    assert plan(GB300, 262144, 1 << 28, 15, hot_bin=7, kernel=pkg.KERNEL_DIRECT)["hot_bin"] == -1
    for bad in (262144, 10 ** 6):
        with pytest.raises(pkg.DsmemHistError) as e:
            plan(GB300, 262144, 1 << 28, 15, hot_bin=bad)
        assert e.value.code == pkg.DSMEM_HIST_EINVAL


def test_planner_helper_row():
    """The helper kernel gets a partial row of its own for single-pass ship
    plans of at least 2^24 keys without a hot bin that leave SMs idle."""
    rows = lambda p: (p["partial_rows"], p["workspace_bytes"])
    p = plan(GB300, 262144, 1 << 28, 15, cluster_size=8)   # 15 clusters of 8: 32 SMs idle
    assert p["num_clusters"] == 15 and rows(p) == (16, 16 * 262144 * 4 + 32)
    r = plan(GB300, 524288, 1 << 30, 7, cluster_size=16)   # 7 clusters of 16: 40 SMs idle
    assert rows(r) == (8, 8 * 524288 * 4 + 32)
    small = plan(GB300, 262144, (1 << 24) - 1, 15, cluster_size=8)
    assert small["partial_rows"] == small["num_clusters"]  # too few keys
    assert plan(GB300, 262144, 1 << 24, 15, cluster_size=8)["partial_rows"] == 16
    full = plan(GB300, 65536, 1 << 26, 76, cluster_size=2)  # 76 clusters of 2: no SM idle
    assert full["partial_rows"] == full["num_clusters"] == 76
    multi = plan(GB300, 1 << 22, 1 << 28, 0, cluster_size=16)
    assert multi["passes"] > 1 and multi["partial_rows"] == multi["num_clusters"]
    hot = plan(GB300, 262144, 1 << 28, 15, cluster_size=8, hot_bin=5)
    assert rows(hot) == rows(p)                            # the hot-bin kernel takes it too
    direct = plan(GB300, 262144, 1 << 28, 15, cluster_size=8, kernel=pkg.KERNEL_DIRECT)
    assert direct["partial_rows"] == direct["num_clusters"]
