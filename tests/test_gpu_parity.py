"""GPU parity: the CUDA library, called through its C ABI, against the CPU
oracle, bit for bit (integer counts: one correct answer).

Covers the pins, forced launch shapes (every cluster size, both aggregation
modes, block sizes, misaligned key pointers, ragged lengths), multi-pass bin
ranges, the five synthetic workloads at full size in the launch
configuration the benchmark times, the global-atomics comparison kernel, the
host-buffer entry point and concurrent streams.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import cluster_distributed_shared_gb300 as pkg  # noqa: E402
import gen  # noqa: E402
import oracle  # noqa: E402
from tests import pins  # noqa: E402

pytestmark = pytest.mark.gpu

# Cluster size each synthetic workload is published with.
WORKLOAD_CLUSTER = {
    "uniform-1M-8K": 2,
    "uniform-64M-64K": 2,
    "uniform-256M-256K": 8,
    "zipf1.1-256M-256K": 8,
    "runs256-1G-512K": 16,
}


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.init()
    yield
    torch.cuda.synchronize()


def to_np(t):
    return t.cpu().numpy().view(np.uint32)


def gpu_hist(keys, num_bins, out=None, **kw):
    d = torch.from_numpy(np.ascontiguousarray(keys, np.int32)).cuda()
    o = None
    if out is not None:
        o = torch.from_numpy(out.view(np.int32)).cuda()
    r = pkg.dsmem_hist(d, num_bins, out=o, **kw)
    torch.cuda.synchronize()
    return to_np(r)


def forced(**kw):
    return lambda keys, num_bins, out=None: gpu_hist(keys, num_bins, out, **kw)


def global_atomic(keys, num_bins, out=None):
    d = torch.from_numpy(np.ascontiguousarray(keys, np.int32)).cuda()
    o = None if out is None else torch.from_numpy(out.view(np.int32)).cuda()
    r = pkg.dsmem_hist_global_atomic(d, num_bins, out=o)
    torch.cuda.synchronize()
    return to_np(r)


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pins_default_plan(pin):
    pin(gpu_hist)


D, SH = pkg.KERNEL_DIRECT, pkg.KERNEL_SHIP


@pytest.mark.parametrize("shape", [
    dict(cluster_size=1, aggregate=0), dict(cluster_size=2, aggregate=1, kernel=D),
    dict(cluster_size=4, aggregate=0, block_threads=256), dict(cluster_size=8, aggregate=1, kernel=D),
    dict(cluster_size=16, aggregate=0, kernel=D), dict(cluster_size=16, aggregate=1, block_threads=64),
    dict(cluster_size=2, kernel=SH), dict(cluster_size=3, kernel=SH), dict(cluster_size=8, kernel=SH),
    dict(cluster_size=16, kernel=SH), dict(cluster_size=5, kernel=SH, num_clusters=1),
], ids=str)
@pytest.mark.parametrize("pin", [pins.pin_brute_force_tiny, pins.pin_cycle,
                                 pins.pin_constructed_counts, pins.pin_single_value,
                                 pins.pin_out_of_range, pins.pin_overwrite, pins.pin_empty],
                         ids=lambda p: p.__name__)
def test_pins_forced_shapes(pin, shape):
    pin(forced(**shape))


@pytest.mark.parametrize("pin", [pins.pin_brute_force_tiny, pins.pin_cycle,
                                 pins.pin_single_value, pins.pin_out_of_range,
                                 pins.pin_overwrite, pins.pin_empty], ids=lambda p: p.__name__)
def test_pins_global_atomic(pin):
    pin(global_atomic)


@pytest.mark.parametrize("num_bins", [8192, 65536, 100003, 262144, 524288])
def test_forced_shape_sweep(num_bins):
    n = 5_000_003
    base = gen.uniform(n + 3, num_bins + num_bins // 16, seed=num_bins)  # ~6% out of range
    base[::1001] = -7
    dev = torch.from_numpy(base).cuda()
    for off in (0, 3):
        keys_np = base[off:off + n]
        want = oracle.histogram(keys_np, num_bins)
        keys = dev[off:off + n]
        shapes = [dict(cluster_size=P, kernel=D, aggregate=agg, block_threads=t)
                  for P in (1, 2, 4, 8, 16) for agg in (0, 1) for t in (256, 1024)]
        shapes += [dict(cluster_size=P, kernel=SH) for P in (2, 3, 4, 6, 8, 12, 16)]
        for kw in shapes:
            got = pkg.dsmem_hist(keys, num_bins, **kw)
            torch.cuda.synchronize()
            g = to_np(got)
            assert np.array_equal(g, want), (num_bins, off, kw, np.flatnonzero(g != want)[:8])


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 31, 32, 33, 127, 128, 129, 130, 511, 4099, 65537,
                               2 * 128 * 32 * 6 + 5, 1 << 20])
def test_ragged_small_lengths(n):
    num_bins = 37
    base = gen.uniform(n + 3, 40, seed=n)
    dev = torch.from_numpy(base).cuda()
    for off in (0, 1, 2, 3):
        want = oracle.histogram(base[off:off + n], num_bins)
        for kw in (dict(kernel=D, aggregate=0), dict(kernel=D, aggregate=1), dict(kernel=SH)):
            got = pkg.dsmem_hist(dev[off:off + n], num_bins, cluster_size=2, num_clusters=3, **kw)
            torch.cuda.synchronize()
            assert np.array_equal(to_np(got), want), (n, off, kw)


def test_ship_overflow_and_runs_paths():
    # Keys that all belong to one owner overflow its staging columns (remote
    # increments take over); runs of equal keys take the whole-tile path;
    # partial runs and run boundaries mix both.
    rng = np.random.default_rng(3)
    n = 1 << 22
    cases = []
    cases.append((rng.integers(0, 32768, n).astype(np.int32), 262144, 8))      # owner 0 only
    cases.append((rng.integers(7 * 32768, 8 * 32768, n).astype(np.int32), 262144, 8))  # last owner
    runs = np.repeat(rng.integers(0, 524288, n // 128), 128).astype(np.int32)
    cases.append((runs, 524288, 16))
    odd = np.repeat(rng.integers(0, 65536, n // 37 + 1), 37)[:n].astype(np.int32)
    cases.append((odd, 65536, 2))
    mix = rng.integers(0, 262144, n).astype(np.int32)
    mix[: n // 2] = 12345                                                       # one hot bin
    cases.append((mix, 262144, 8))
    for keys, num_bins, P in cases:
        want = oracle.histogram(keys, num_bins)
        for kw in (dict(kernel=SH), dict(kernel=D)):
            got = gpu_hist(keys, num_bins, cluster_size=P, **kw)
            assert np.array_equal(got, want), (num_bins, P, kw)


def test_ship_run_tiles_pairs_and_boundaries():
    # The ship kernel deals each warp two consecutive 128-key tiles per round
    # and turns a run tile followed by a run tile of the same key into one
    # remote red of 256.  Built per 128-key tile: pairs of equal run tiles,
    # run tiles with different keys side by side, runs that straddle a pair
    # (odd-aligned runs of 256), runs of keys outside the bins, run tiles next
    # to ordinary tiles; at several pointer offsets (the tiles then start
    # mid-run) and in a multi-pass shape.
    rng = np.random.default_rng(11)
    ntiles = 1 << 14
    kinds = rng.integers(0, 6, ntiles // 2)
    tiles = []
    for kind in kinds:
        a, b = rng.integers(0, 262144, 2)
        if kind == 0:     # one run of 256 on the pair
            tiles += [np.full(128, a), np.full(128, a)]
        elif kind == 1:   # two runs of 128, different keys
            tiles += [np.full(128, a), np.full(128, b)]
        elif kind == 2:   # run then ordinary tile
            tiles += [np.full(128, a), rng.integers(0, 262144, 128)]
        elif kind == 3:   # ordinary tile then run
            tiles += [rng.integers(0, 262144, 128), np.full(128, a)]
        elif kind == 4:   # runs of keys no bin holds (dropped), one negative
            tiles += [np.full(128, 262144 + a), np.full(128, -1 - a)]
        else:             # a run of 256 shifted by one tile: straddles two pairs
            tiles += [np.full(128, b), np.full(128, a)]
    keys = np.concatenate(tiles).astype(np.int32)
    # kind 5 pairs end with key a; let the next pair start with the same key
    # where it is also a run, so some runs of 256 start at an odd tile.
    for t in range(1, ntiles - 1, 2):
        if kinds[t // 2] == 5 and t + 1 < ntiles and rng.random() < 0.5:
            keys[(t + 1) * 128:(t + 2) * 128] = keys[t * 128]
    for off in (0, 1, 3):
        k = keys[off:]
        for num_bins, P in ((262144, 8), (524288, 16)):
            want = oracle.histogram(k, num_bins)
            got = gpu_hist(k, num_bins, cluster_size=P, kernel=SH)
            assert np.array_equal(got, want), (off, num_bins, P)
    # Eight passes of 32768 bins each: most runs hold keys of another pass.
    want = oracle.histogram(keys, 262144)
    plan = pkg.dsmem_hist_plan(262144, keys.size, cluster_size=2, kernel=SH,
                               max_slice_bytes=4 * 16384)
    assert plan["passes"] == 8 and plan["kernel"] == SH
    got = gpu_hist(keys, 262144, cluster_size=2, kernel=SH, max_slice_bytes=4 * 16384)
    assert np.array_equal(got, want)


def test_ship_mostly_out_of_range_and_multi_pass():
    # Keys outside the pass meet the always-full cursor row and leave through
    # the spill path on almost every tile; later passes subtract their base.
    rng = np.random.default_rng(11)
    n = 3_000_017
    num_bins = 262144
    keys = rng.integers(-2 ** 31, 2 ** 31 - 1, n, dtype=np.int64).astype(np.int32)
    keys[::10] = rng.integers(0, num_bins, keys[::10].size)               # 10% in range
    want = oracle.histogram(keys, num_bins)
    for P in (3, 8, 16):
        got = gpu_hist(keys, num_bins, cluster_size=P, kernel=SH)
        assert np.array_equal(got, want), P
    for num_bins, P in [(1 << 21, 8), (600_001, 4), (1 << 20, 2)]:
        keys = gen.uniform(n, num_bins + 1000, seed=num_bins)
        plan = pkg.dsmem_hist_plan(num_bins, n, cluster_size=P, kernel=SH)
        assert plan["kernel"] == SH and plan["passes"] > 1, plan
        got = gpu_hist(keys, num_bins, cluster_size=P, kernel=SH)
        assert np.array_equal(got, oracle.histogram(keys, num_bins)), (num_bins, P)


def test_multi_pass_bin_ranges():
    n = 3_000_001
    for num_bins, kw in [(1 << 22, {}), (100003, dict(max_slice_bytes=4096)),
                         (929792, dict(max_slice_bytes=232448, cluster_size=16)),
                         (1 << 21, dict(cluster_size=2, aggregate=0))]:
        keys = gen.uniform(n, num_bins, seed=num_bins)
        plan = pkg.dsmem_hist_plan(num_bins, n, **kw)
        got = gpu_hist(keys, num_bins, **kw)
        assert np.array_equal(got, oracle.histogram(keys, num_bins)), (num_bins, plan)
    assert pkg.dsmem_hist_plan(1 << 22, n)["passes"] > 1


def test_max_slice_single_pass():
    # Largest slice a CTA can opt in to, with the largest cluster.
    plan = pkg.dsmem_hist_plan(929792, 1 << 24, cluster_size=16, max_slice_bytes=232448)
    assert plan["passes"] == 1 and plan["smem_bytes"] == 232448
    keys = gen.uniform(1 << 24, 1 << 20, seed=4)
    got = gpu_hist(keys, 929792, cluster_size=16, max_slice_bytes=232448)
    assert np.array_equal(got, oracle.histogram(keys, 929792))


def _full_workload(name, seed):
    keys = gen.workload(name, seed)
    num_bins = gen.WORKLOADS[name]["num_bins"]
    return keys, num_bins


@pytest.mark.parametrize("name,seed", [(w, s) for w in WORKLOAD_CLUSTER for s in (0, 1, 2)] +
                         [(w, s) for w in ("uniform-1M-8K", "uniform-64M-64K") for s in range(3, 10)])
def test_workload_full_size(name, seed):
    keys, num_bins = _full_workload(name, seed)
    want = oracle.histogram(keys, num_bins)
    assert int(want.sum(dtype=np.uint64)) == keys.size  # every generated key is in range
    d = torch.from_numpy(keys).cuda()
    del keys
    P = WORKLOAD_CLUSTER[name]
    plan = pkg.dsmem_hist_plan(num_bins, d.numel(), cluster_size=P)
    assert plan["cluster_size"] == P and plan["bins_per_cta"] == num_bins // P
    assert plan["passes"] == 1
    out = torch.full((num_bins,), -1, dtype=torch.int32, device="cuda")
    for kw in (dict(cluster_size=P), {}):   # the benchmark's shape, then the planner's
        pkg.dsmem_hist(d, num_bins, out=out, **kw)
        torch.cuda.synchronize()
        got = to_np(out)
        assert np.array_equal(got, want), (name, seed, kw, np.flatnonzero(got != want)[:8])
    assert plan["kernel"] == SH
    if seed == 0:
        pkg.dsmem_hist_global_atomic(d, num_bins, out=out)
        torch.cuda.synchronize()
        assert np.array_equal(to_np(out), want)
        for agg in (0, 1):
            pkg.dsmem_hist(d, num_bins, out=out, cluster_size=P, kernel=D, aggregate=agg)
            torch.cuda.synchronize()
            assert np.array_equal(to_np(out), want), agg
    del d
    torch.cuda.empty_cache()


def test_host_entry_point():
    num_bins = 262144
    for n in (0, 1, 4099, (1 << 24) + 12345, 3 * (1 << 24) + 7):
        keys = gen.uniform(n, num_bins, seed=n)
        want = oracle.histogram(keys, num_bins)
        got = pkg.dsmem_hist_host(keys, num_bins)                 # pageable numpy
        assert np.array_equal(got, want), n
        pinned = torch.from_numpy(keys).pin_memory()
        out = torch.empty(num_bins, dtype=torch.int32).pin_memory()
        pkg.dsmem_hist_host(pinned, num_bins, out=out)             # pinned torch
        assert np.array_equal(out.numpy().view(np.uint32), want), n


def test_two_streams_do_not_share_scratch():
    num_bins = 262144
    a_np = gen.uniform(1 << 24, num_bins, seed=21)
    b_np = gen.zipf(1 << 24, num_bins, seed=22)
    want_a, want_b = oracle.histogram(a_np, num_bins), oracle.histogram(b_np, num_bins)
    a, b = torch.from_numpy(a_np).cuda(), torch.from_numpy(b_np).cuda()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    torch.cuda.synchronize()
    for i in range(6):
        with torch.cuda.stream(sa):
            outs.append(("a", pkg.dsmem_hist(a, num_bins, stream=sa)))
        with torch.cuda.stream(sb):
            outs.append(("b", pkg.dsmem_hist(b, num_bins, stream=sb)))
    torch.cuda.synchronize()
    for tag, o in outs:
        assert np.array_equal(to_np(o), want_a if tag == "a" else want_b)


def test_repeat_is_deterministic_across_shapes():
    num_bins = 65536
    keys = gen.zipf(1 << 22, num_bins, seed=5)
    want = oracle.histogram(keys, num_bins)
    d = torch.from_numpy(keys).cuda()
    for i in range(5):
        for kw in (dict(cluster_size=2), dict(cluster_size=4, num_clusters=1),
                   dict(cluster_size=8, num_clusters=64), dict(kernel=D, aggregate=0),
                   dict(kernel=D, aggregate=1), dict(kernel=SH, cluster_size=16, num_clusters=40)):
            got = pkg.dsmem_hist(d, num_bins, **kw)
            torch.cuda.synchronize()
            assert np.array_equal(to_np(got), want), kw


@pytest.mark.parametrize("P", [2, 4, 8, 16])
@pytest.mark.parametrize("kpt", [8, 4])
def test_long_round_chains_in_one_cluster(P, kpt):
    # One cluster of the ship kernel walks hundreds of rounds, so every
    # buffer, cursor set and mbarrier phase is reused many times; Zipf keys
    # make the owners' loads uneven from round to round, and the length
    # leaves a ragged tail.
    num_bins = P * 32768
    n = (1 << 23) + 12345
    keys_np = gen.zipf(n, num_bins, seed=40 + P)
    want = oracle.histogram(keys_np, num_bins)
    keys = torch.from_numpy(keys_np).cuda()
    plan = pkg.dsmem_hist_plan(num_bins, n, cluster_size=P, kernel=SH, num_clusters=1)
    plan["keys_per_thread"] = kpt
    rounds = n // (P * pkg.SHIP_THREADS * kpt)
    assert plan["num_clusters"] == 1 and plan["bins_per_cta"] == 32768 and rounds >= 70
    partials = torch.empty(-(-plan["workspace_bytes"] // 4), dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream()
    for _ in range(3):
        pkg.dsmem_hist_partials(keys, num_bins, plan, partials, 0, s)
        bins = pkg.dsmem_hist_reduce(partials, plan["partial_rows"], plan["partial_stride"], num_bins,
                                     stream=s)
        torch.cuda.synchronize()
        assert np.array_equal(to_np(bins), want)
    assert pkg.dsmem_hist_device_status() == 0


def test_errors_on_device():
    d = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(pkg.DsmemHistError) as e:
        pkg.dsmem_hist(d, 100, cluster_size=17)
    assert e.value.code == pkg.DSMEM_HIST_EINVAL
    with pytest.raises(pkg.DsmemHistError):
        pkg.dsmem_hist(d, 100, block_threads=48)
    with pytest.raises(TypeError):
        pkg.dsmem_hist(d.cpu(), 100)
    # the library stays usable after rejected calls
    got = pkg.dsmem_hist(d, 100)
    torch.cuda.synchronize()
    want = np.zeros(100, np.uint32)
    want[0] = 16
    assert np.array_equal(to_np(got), want)


def test_plan_on_device_confirms_cluster_16():
    p = pkg.dsmem_hist_plan(524288, 1 << 30)
    assert p["cluster_size"] == 16 and p["max_active_clusters"] >= 1
    p8 = pkg.dsmem_hist_plan(262144, 1 << 28)
    assert p8["cluster_size"] == 8 and p8["max_active_clusters"] >= 1
    assert p8["num_clusters"] == p8["max_active_clusters"]


def test_randomized_shapes_and_inputs():
    # Seeded random trials over bin counts, lengths, misaligned starts, forced
    # cluster sizes and kernels, and key mixes (negatives, out of range,
    # runs, one hot bin); every result bit-exact against the oracle.
    rng = np.random.default_rng(2024)
    for trial in range(60):
        num_bins = int(rng.choice([1, 7, 100, 4096, 8191, 40000, 65536, 131072, 262144, 300007]))
        n = int(rng.integers(0, 3_000_000))
        off = int(rng.integers(0, 4))
        keys = rng.integers(-num_bins // 8 - 2, num_bins + num_bins // 8 + 2, n + off).astype(np.int32)
        if trial % 3 == 0 and n > 1024:                      # runs of equal keys
            starts = rng.integers(0, n - 512, 16)
            for s0 in starts:
                keys[s0:s0 + 512] = rng.integers(0, num_bins)
        if trial % 4 == 1 and n > 0:                         # one hot bin
            keys[rng.random(n + off) < 0.2] = rng.integers(0, num_bins)
        P = int(rng.choice([0, 2, 3, 4, 8, 16]))
        kw = {}
        if P:
            kw["cluster_size"] = P
        if P >= 2 and trial % 2 == 0:
            kw["kernel"] = SH
        elif P and trial % 5 == 0:
            kw["kernel"] = D
        sub = keys[off:off + n]
        want = oracle.histogram(sub, num_bins)
        dev = torch.from_numpy(keys).cuda()[off:off + n]
        got = pkg.dsmem_hist(dev, num_bins, **kw)
        torch.cuda.synchronize()
        g = to_np(got)
        assert np.array_equal(g, want), (trial, num_bins, n, off, kw, np.flatnonzero(g != want)[:8])


def test_environment_overrides_fill_open_request_fields(monkeypatch):
    monkeypatch.setenv("DSMEM_HIST_KERNEL", "0")
    monkeypatch.setenv("DSMEM_HIST_CLUSTER", "4")
    p = pkg.dsmem_hist_plan(262144, 1 << 24)
    assert p["kernel"] == D and p["cluster_size"] == 4
    forced = pkg.dsmem_hist_plan(262144, 1 << 24, cluster_size=8, kernel=SH)
    assert forced["kernel"] == SH and forced["cluster_size"] == 8   # explicit fields win
    keys = gen.uniform(1 << 20, 262144, seed=12)
    assert np.array_equal(gpu_hist(keys, 262144), oracle.histogram(keys, 262144))


@pytest.mark.parametrize("share", [0.0, 0.25, 0.6])
def test_hot_bin_hint_is_exact(share):
    """The hinted ship kernel (the hot bin's keys counted per thread instead of
    staged) against the oracle: with and without the hint, a hint on a bin
    that is not hot, at P = 8 and P = 2, and across passes."""
    n, num_bins = 1 << 24, 262144
    keys = gen.hot(n, num_bins, seed=61, share=share)
    hb = gen.hot_bin(num_bins, 61)
    keys[:5] = [-1, num_bins, 2 ** 31 - 1, -2 ** 31, hb]   # out-of-range keys ride along
    keys[1000:1128] = hb                                     # a whole tile of the hot bin
    want = oracle.histogram(keys, num_bins)
    d = torch.from_numpy(keys).cuda()
    for kw in (dict(cluster_size=8), dict(cluster_size=8, hot_bin=hb), dict(cluster_size=8, hot_bin=3),
               dict(cluster_size=2, hot_bin=hb), dict(cluster_size=16, hot_bin=hb),
               dict(cluster_size=8, hot_bin=hb, num_clusters=3)):
        got = to_np(pkg.dsmem_hist(d, num_bins, **kw))
        torch.cuda.synchronize()
        assert np.array_equal(got, want), (share, kw, np.flatnonzero(got != want)[:8])
    plan = pkg.dsmem_hist_plan(num_bins, n, cluster_size=2, hot_bin=hb)
    assert plan["hot_bin"] == hb and plan["passes"] == 4   # the hot bin lies in one of four passes
    # through the two-stage entry points with the hinted plan
    partials = torch.empty(-(-plan["workspace_bytes"] // 4), dtype=torch.int32,
                           device="cuda")
    pkg.dsmem_hist_partials(d, num_bins, plan, partials)
    got = to_np(pkg.dsmem_hist_reduce(partials, plan["partial_rows"], plan["partial_stride"],
                                      num_bins))
    torch.cuda.synchronize()
    assert np.array_equal(got, want)


def test_hot_workload_full_size_with_and_without_hint():
    keys, num_bins = _full_workload("hot25-256M-256K", 0)
    want = oracle.histogram(keys, num_bins)
    hb = gen.hot_bin(num_bins, 0)
    assert want.argmax() == hb
    d = torch.from_numpy(keys).cuda()
    del keys
    out = torch.full((num_bins,), -1, dtype=torch.int32, device="cuda")
    for kw in (dict(cluster_size=8), dict(cluster_size=8, hot_bin=hb)):
        pkg.dsmem_hist(d, num_bins, out=out, **kw)
        torch.cuda.synchronize()
        assert np.array_equal(to_np(out), want), kw
    del d
    torch.cuda.empty_cache()


_AUTO_SCRIPT = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
import cluster_distributed_shared_gb300 as pkg, gen, oracle
n, nb = 1 << 24, 262144
hot = gen.hot(n, nb, seed=81, share=0.25)
uni = gen.uniform(n, nb, seed=82)
s = torch.cuda.Stream()
for tag, keys in [("hot1", hot), ("hot2", hot), ("hot3", hot), ("uni1", uni), ("uni2", uni),
                  ("hot4", hot), ("hot5", hot)]:
    d = torch.from_numpy(keys).cuda()
    torch.cuda.synchronize()
    print("CALL", tag, file=sys.stderr, flush=True)
    got = pkg.dsmem_hist(d, nb, stream=s)      # automatic choice
    s.synchronize()
    ok = np.array_equal(got.cpu().numpy().view(np.uint32), oracle.histogram(keys, nb))
    print("PARITY", tag, ok, file=sys.stderr, flush=True)
# the caller can turn the choice off
d = torch.from_numpy(hot).cuda()
print("CALL off", file=sys.stderr, flush=True)
got = pkg.dsmem_hist(d, nb, stream=s, hot_bin=-1)
s.synchronize()
print("PARITY off", np.array_equal(got.cpu().numpy().view(np.uint32), oracle.histogram(hot, nb)),
      file=sys.stderr, flush=True)
print("HOTBIN", gen.hot_bin(nb, 81), file=sys.stderr, flush=True)
"""


def test_hot_bin_kernel_is_chosen_from_the_previous_histogram():
    """A bin with a quarter of the keys makes the next call on the same stream
    take the hot-bin kernel; uniform keys switch it off again; every call is
    exact."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, DSMEM_HIST_TRACE="1")
    out = subprocess.run([sys.executable, "-c", _AUTO_SCRIPT, root], env=env, capture_output=True,
                         text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = out.stderr.splitlines()
    hot_bin = int([l for l in lines if l.startswith("HOTBIN")][0].split()[1])
    chose, current = {}, None
    for l in lines:
        if l.startswith("CALL"):
            current = l.split()[1]
            chose[current] = None
        elif "-> hot-bin kernel" in l and current is not None:
            chose[current] = int(l.split("bin ")[1].split()[0])
        elif l.startswith("PARITY"):
            assert l.split()[2] == "True", l
    assert chose["hot1"] is None                        # nothing known yet
    assert chose["hot2"] == chose["hot3"] == hot_bin    # the previous call had the hot bin
    assert chose["uni1"] == hot_bin                     # chosen from the hot call before it
    assert chose["uni2"] is None                        # uniform keys report no hot bin
    assert chose["hot4"] is None and chose["hot5"] == hot_bin
    assert chose["off"] is None


@pytest.mark.parametrize("mode,share", [("0", None), ("1", None), ("1", "0"), ("1", "0.5"),
                                        ("1", "1")])
def test_idle_sm_helper_and_mop_up(monkeypatch, mode, share):
    """Clusters of 8 leave 32 SMs idle; a global-atomic helper kernel on them
    takes the tiles after the clusters' rounds, and a mop-up kernel after the
    cluster kernel takes the ones it has not claimed.  Exact with the helper
    off, at its planned share, with no tiles for it, with half and with all
    of them (the mop-up then does much of the work): on uniform, Zipf and
    run-heavy keys, at a pointer offset, through the product call, the
    two-stage entry points (accumulating too) and the host entry point."""
    monkeypatch.setenv("DSMEM_HIST_HELPER", mode)
    if share is not None:
        monkeypatch.setenv("DSMEM_HIST_HELPER_SHARE", share)
    num_bins = 262144
    n = (1 << 25) + 1001
    cases = [gen.uniform(n, num_bins, seed=81), gen.zipf(n, num_bins, seed=82),
             gen.workload("runs256-1G-512K", 83, n=1 << 25) % num_bins]
    for keys in cases:
        keys = np.ascontiguousarray(keys, np.int32)
        want = oracle.histogram(keys, num_bins)
        assert np.array_equal(gpu_hist(keys, num_bins, cluster_size=8), want)
        d = torch.from_numpy(keys).cuda()
        sub = d[3:]                                          # 12-byte offset: a scalar head
        want_sub = oracle.histogram(keys[3:], num_bins)
        out = torch.empty(num_bins, dtype=torch.int32, device="cuda")
        pkg.dsmem_hist(sub, num_bins, out=out, cluster_size=8)
        torch.cuda.synchronize()
        assert np.array_equal(to_np(out), want_sub)
        plan = pkg.dsmem_hist_plan(num_bins, sub.numel(), cluster_size=8)
        assert plan["kernel"] == SH and plan["passes"] == 1
        assert plan["partial_rows"] == plan["num_clusters"] + (mode != "0")
        partials = torch.empty(-(-plan["workspace_bytes"] // 4), dtype=torch.int32, device="cuda")
        half = (sub.numel() // 2) & ~127
        pkg.dsmem_hist_partials(sub[:half], num_bins, plan, partials, 0)
        pkg.dsmem_hist_partials(sub[half:], num_bins, plan, partials, 1)
        got = to_np(pkg.dsmem_hist_reduce(partials, plan["partial_rows"], plan["partial_stride"],
                                          num_bins, out))
        assert np.array_equal(got, want_sub)
        assert np.array_equal(pkg.dsmem_hist_host(keys, num_bins), want)
        del d, sub
    assert pkg.dsmem_hist_device_status() == 0


@pytest.mark.parametrize("seed", [4242, 777])
def test_helper_randomized_streams(seed):
    """Seeded random launches that take the idle-SM helper (single-pass
    plans of clusters of 8 or 16 with at least 2^24 keys), issued back to back
    on three streams with no synchronisation between them, so that helpers,
    mop-ups and share reports of neighbouring launches overlap: random bin
    counts, lengths with ragged tails, misaligned starts, key mixes (uniform,
    Zipf, runs, one hot bin, out-of-range keys), the product call and the two
    stages (accumulating); every result bit-exact against the oracle."""
    rng = np.random.default_rng(seed)
    streams = [torch.cuda.Stream() for _ in range(3)]
    shapes = [(8192, 8), (100003, 8), (200000, 8), (262144, 8), (262144, 0), (300007, 16),
              (524288, 16)]
    trials = []
    for trial in range(21):
        num_bins, P = shapes[trial % len(shapes)]
        n = (1 << 24) + int(rng.integers(0, 1 << 22))
        off = int(rng.integers(0, 4))
        kseed = seed + 500 + trial
        mix = int(rng.integers(0, 5))
        if mix == 0:
            keys = gen.uniform(n + off, num_bins, seed=kseed)
        elif mix == 1:
            keys = gen.zipf(n + off, num_bins, seed=kseed)
        elif mix == 2:
            keys = gen.runs(n + off, num_bins, seed=kseed)
        elif mix == 3:
            keys = gen.hot(n + off, num_bins, seed=kseed)
        else:
            keys = gen.uniform(n + off, num_bins + num_bins // 4, seed=kseed) - num_bins // 8
        keys = np.ascontiguousarray(keys, np.int32)
        plan = pkg.dsmem_hist_plan(num_bins, n, **({"cluster_size": P} if P else {}))
        assert plan["passes"] == 1 and plan["partial_rows"] == plan["num_clusters"] + 1, plan
        trials.append((trial, num_bins, P, off, keys, plan))
    dev = [torch.from_numpy(t[4]).cuda() for t in trials]
    torch.cuda.synchronize()                 # keys uploaded before the side streams read them
    results = []
    for (trial, num_bins, P, off, keys, plan), d in zip(trials, dev):
        s = streams[trial % len(streams)]
        sub = d[off:]
        kw = {"cluster_size": P} if P else {}
        if trial % 3 == 2:                   # the two stages, the second accumulating
            partials = torch.empty(-(-plan["workspace_bytes"] // 4), dtype=torch.int32,
                                   device="cuda")
            cut = int(rng.integers(1, sub.numel()))
            pkg.dsmem_hist_partials(sub[:cut], num_bins, plan, partials, 0, stream=s)
            pkg.dsmem_hist_partials(sub[cut:], num_bins, plan, partials, 1, stream=s)
            got = pkg.dsmem_hist_reduce(partials, plan["partial_rows"], plan["partial_stride"],
                                        num_bins, stream=s)
            results.append((got, partials))
        else:
            results.append((pkg.dsmem_hist(sub, num_bins, stream=s, **kw), None))
    torch.cuda.synchronize()
    for (trial, num_bins, P, off, keys, plan), (got, _) in zip(trials, results):
        want = oracle.histogram(keys[off:], num_bins)
        g = to_np(got)
        assert np.array_equal(g, want), (trial, num_bins, P, off, np.flatnonzero(g != want)[:8])
    assert pkg.dsmem_hist_device_status() == 0


_SHARE_SCRIPT = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
import cluster_distributed_shared_gb300 as pkg, gen, oracle
n, nb = 1 << 26, 262144
for name, keys in [("zipf", gen.zipf(n, nb, seed=91)), ("uniform", gen.uniform(n, nb, seed=92))]:
    want = oracle.histogram(keys, nb)
    d = torch.from_numpy(keys).cuda()
    s = torch.cuda.Stream()
    print("WORKLOAD", name, file=sys.stderr, flush=True)
    for i in range(8):
        got = pkg.dsmem_hist(d, nb, stream=s, cluster_size=8)
        s.synchronize()                      # the next call reads this one's report
        ok = np.array_equal(got.cpu().numpy().view(np.uint32), want)
        print("PARITY", name, i, ok, file=sys.stderr, flush=True)
"""


def test_helper_share_follows_the_reports():
    """The helper's share starts from the idle SMs' expected pace and then
    follows each launch's report on the same stream: on Zipf keys (its cache
    counts the frequent keys in shared memory) it grows well past the prior,
    on uniform keys (a fresh stream) it settles near the prior; every call is
    exact."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, DSMEM_HIST_TRACE="1")
    out = subprocess.run([sys.executable, "-c", _SHARE_SCRIPT, root], env=env, capture_output=True,
                         text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-3000:]
    shares, current = {}, None
    for l in out.stderr.splitlines():
        if l.startswith("WORKLOAD"):
            current = l.split()[1]
            shares[current] = []
        elif l.startswith("PARITY"):
            assert l.split()[3] == "True", l
        elif "reports share" in l and current is not None:
            # "... reports share T -> share BEFORE -> AFTER"
            parts = l.split("->")
            shares[current].append((float(parts[1].split()[1]), float(parts[2])))
    for name in ("zipf", "uniform"):
        assert len(shares[name]) >= 6, shares            # one report per call after the first
        prior = shares[name][0][0]
        assert 0.05 < prior < 0.2                         # idle SMs x pace / all SMs
        assert all(0.01 <= after <= 0.6 for _, after in shares[name])
    assert shares["zipf"][-1][1] > 1.5 * shares["zipf"][0][0]
    assert 0.5 * shares["uniform"][0][0] < shares["uniform"][-1][1] < 2.0 * shares["uniform"][0][0]
