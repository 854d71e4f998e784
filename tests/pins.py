"""Pins for any histogram implementation `hist(keys, num_bins, out=None)`.

Each pin checks the result against something fixed independently of the
implementation under test: brute force on tiny inputs, inputs built with
known per-bin counts (closed form), invariants, and numpy's bincount on the
in-range keys.  The definition being pinned ("Distributed Shared Memory",
section "The cluster histogram", with the readings stated in the oracle):

    bins[b] = #{ i : keys[i] == b } mod 2^32 for 0 <= b < num_bins;
    keys outside [0, num_bins) are not counted; `bins` is overwritten.

The same pins run against the CPU oracle (tests/test_oracle.py) and, on a GPU,
against the CUDA library; tests/test_oracle.py also shows that each planted
mistake (off-by-one bound, negative keys wrapped, no zeroing, a dropped key,
a shifted bin, deduplicated keys, narrow counters) fails at least one pin.
"""
from __future__ import annotations

import numpy as np

INT32_MIN = -(2**31)
INT32_MAX = 2**31 - 1


def _rng(seed):
    return np.random.default_rng(seed)


def brute_force(keys: np.ndarray, num_bins: int) -> np.ndarray:
    """O(n * B): compare every key with every bin id."""
    keys = np.asarray(keys, dtype=np.int64)
    ids = np.arange(num_bins, dtype=np.int64)
    return (keys[:, None] == ids[None, :]).sum(axis=0).astype(np.uint32)


def pin_brute_force_tiny(hist):
    for seed in range(12):
        r = _rng(seed)
        num_bins = int(r.integers(1, 65))
        n = int(r.integers(0, 4097))
        keys = r.integers(-3, num_bins + 3, size=n).astype(np.int32)
        if n:
            pos = r.integers(0, n, size=min(n, 8))
            keys[pos] = r.choice([INT32_MIN, INT32_MAX, -1, num_bins, 0, num_bins - 1],
                                 size=pos.size)
        got = hist(keys, num_bins)
        assert got.dtype == np.uint32 and got.shape == (num_bins,)
        np.testing.assert_array_equal(got, brute_force(keys, num_bins))


def pin_cycle(hist):
    # keys[i] = i mod B with n = m * B: every bin holds exactly m.
    for num_bins, m in [(1, 5), (7, 3), (64, 17), (4096, 9), (8192, 2)]:
        keys = (np.arange(num_bins * m) % num_bins).astype(np.int32)
        got = hist(keys, num_bins)
        np.testing.assert_array_equal(got, np.full(num_bins, m, np.uint32))


def pin_constructed_counts(hist):
    # Target counts c_b = (7b + 3) mod 11, written out, then shuffled.
    for num_bins, seed in [(1, 0), (11, 1), (97, 2), (1000, 3), (8192, 4)]:
        c = (7 * np.arange(num_bins) + 3) % 11
        keys = np.repeat(np.arange(num_bins), c).astype(np.int32)
        _rng(seed).shuffle(keys)
        np.testing.assert_array_equal(hist(keys, num_bins), c.astype(np.uint32))


def pin_single_value(hist):
    # All keys equal: maximum contention; n above 2^16 catches narrow counters.
    for num_bins, v, n in [(1, 0, 3), (8, 7, 100), (65536, 0, 70001), (65536, 65535, 70001)]:
        keys = np.full(n, v, np.int32)
        want = np.zeros(num_bins, np.uint32)
        want[v] = n
        np.testing.assert_array_equal(hist(keys, num_bins), want)


def pin_out_of_range(hist):
    for num_bins in (1, 5, 4096):
        bad = np.array([-1, num_bins, num_bins + 1, INT32_MIN, INT32_MAX, -num_bins,
                        -(num_bins + 1), INT32_MIN + 1], np.int32)
        np.testing.assert_array_equal(hist(bad, num_bins), np.zeros(num_bins, np.uint32))
        edge = np.array([0, num_bins - 1, num_bins, -1, num_bins - 1], np.int32)
        want = np.zeros(num_bins, np.uint32)
        want[0] += 1
        want[num_bins - 1] += 2
        np.testing.assert_array_equal(hist(edge, num_bins), want)


def pin_empty(hist):
    for num_bins in (1, 3, 8192):
        np.testing.assert_array_equal(hist(np.zeros(0, np.int32), num_bins),
                                      np.zeros(num_bins, np.uint32))


def pin_overwrite(hist):
    # `bins` is overwritten: stale contents of the output must not leak in.
    r = _rng(7)
    for num_bins in (1, 33, 4096):
        keys = r.integers(0, num_bins, size=5000).astype(np.int32)
        out = np.full(num_bins, 0xDEADBEEF, np.uint32)
        got = hist(keys, num_bins, out=out)
        np.testing.assert_array_equal(got, brute_force(keys, num_bins))


def pin_invariants(hist):
    r = _rng(11)
    for num_bins in (2, 257, 8192):
        keys = r.integers(-num_bins // 2, num_bins + num_bins // 2, size=20000).astype(np.int32)
        got = hist(keys, num_bins)
        in_range = (keys >= 0) & (keys < num_bins)
        assert int(got.sum(dtype=np.uint64)) == int(in_range.sum())
        absent = np.setdiff1d(np.arange(num_bins), keys[in_range])
        assert not got[absent].any()
        perm = r.permutation(keys)
        np.testing.assert_array_equal(hist(perm, num_bins), got)


def pin_bincount(hist):
    r = _rng(13)
    for num_bins in (1, 100, 8192, 65536):
        keys = r.integers(-50, num_bins + 50, size=200000).astype(np.int32)
        ok = keys[(keys >= 0) & (keys < num_bins)]
        want = np.bincount(ok, minlength=num_bins).astype(np.uint32)
        np.testing.assert_array_equal(hist(keys, num_bins), want)


ALL_PINS = [
    pin_brute_force_tiny,
    pin_cycle,
    pin_constructed_counts,
    pin_single_value,
    pin_out_of_range,
    pin_empty,
    pin_overwrite,
    pin_invariants,
    pin_bincount,
]
