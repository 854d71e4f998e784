"""The CPU oracle against its pins, and the pins against planted mistakes.

CPU only (no GPU, no CUDA library).
"""
from __future__ import annotations

import json
import os

import numpy as np
import pytest

import gen
import oracle
from tests import pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def oracle_hist(keys, num_bins, out=None):
    return oracle.histogram(keys, num_bins, out=out)


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle_hist)


# --- planted mistakes: every one of them must fail at least one pin --------

def _valid(keys, num_bins):
    keys = np.asarray(keys, np.int64)
    return keys[(keys >= 0) & (keys < num_bins)]


def mutant_inclusive_upper(keys, num_bins, out=None):
    k = np.asarray(keys, np.int64)
    k = k[(k >= 0) & (k <= num_bins)]
    return np.bincount(np.minimum(k, num_bins - 1), minlength=num_bins).astype(np.uint32)


def mutant_negative_wrap(keys, num_bins, out=None):
    k = np.asarray(keys, np.int64) % num_bins  # negatives folded in, like C's % on casts
    k[np.asarray(keys, np.int64) >= num_bins] = -1
    return np.bincount(k[k >= 0], minlength=num_bins).astype(np.uint32)


def mutant_no_zeroing(keys, num_bins, out=None):
    base = out.copy() if out is not None else np.zeros(num_bins, np.uint32)
    return base + np.bincount(_valid(keys, num_bins), minlength=num_bins).astype(np.uint32)


def mutant_drop_last(keys, num_bins, out=None):
    return np.bincount(_valid(np.asarray(keys)[:-1], num_bins), minlength=num_bins).astype(np.uint32)


def mutant_shifted_bin(keys, num_bins, out=None):
    k = _valid(keys, num_bins)
    return np.bincount((k + 1) % num_bins, minlength=num_bins).astype(np.uint32)


def mutant_dedup_runs(keys, num_bins, out=None):
    # counts a run of equal neighbouring keys once (a broken aggregation)
    k = np.asarray(keys, np.int64)
    if k.size:
        k = k[np.concatenate([[True], k[1:] != k[:-1]])]
    return np.bincount(_valid(k, num_bins), minlength=num_bins).astype(np.uint32)


def mutant_u16_counters(keys, num_bins, out=None):
    h = np.bincount(_valid(keys, num_bins), minlength=num_bins)
    return (h.astype(np.uint16)).astype(np.uint32)


MUTANTS = [mutant_inclusive_upper, mutant_negative_wrap, mutant_no_zeroing, mutant_drop_last,
           mutant_shifted_bin, mutant_dedup_runs, mutant_u16_counters]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m.__name__)
def test_pins_reject_mutant(mutant):
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, IndexError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"{mutant.__name__} passed every pin"


# --- golden regression fixtures (written by tests/golden/make_golden.py) -----

def _digest(a: np.ndarray) -> str:
    import hashlib
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


@pytest.mark.parametrize("fixture", sorted(f for f in os.listdir(GOLDEN) if f.endswith(".json")))
def test_golden_fixture(fixture):
    with open(os.path.join(GOLDEN, fixture)) as f:
        g = json.load(f)
    keys = gen.workload(g["workload"], g["seed"]) if "workload" in g else getattr(gen, g["dist"])(
        **g["args"])
    assert _digest(keys) == g["sha256_keys"], "generator output changed"
    bins = oracle.histogram(keys, g["num_bins"])
    assert _digest(bins) == g["sha256_bins"]
    assert int(bins.sum(dtype=np.uint64)) == g["in_range"]
    for b, c in g["sample"]:
        assert int(bins[b]) == c


# --- generator sanity (shape of the synthetic inputs; not parity) -----------

def test_uniform_chi_square():
    keys = gen.uniform(1 << 22, 1024, seed=5)
    h = np.bincount(keys, minlength=1024)
    e = keys.size / 1024
    chi2 = ((h - e) ** 2 / e).sum()
    # 1023 degrees of freedom: mean 1023, sd ~45; 6 sd either side
    assert 750 < chi2 < 1300
    assert keys.min() >= 0 and keys.max() < 1024


def test_uniform_thread_count_invariant():
    a = gen.uniform(3_000_001, 1000, seed=9, threads=1)
    b = gen.uniform(3_000_001, 1000, seed=9, threads=5)
    np.testing.assert_array_equal(a, b)


def test_zipf_shape_closed_form():
    num_bins, s = 262144, 1.1
    cdf, perm = gen.zipf_tables(num_bins, s, seed=0)
    h = np.sum(np.arange(1, num_bins + 1, dtype=np.float64) ** -s)
    assert abs(cdf[0] - 1 / h) < 1e-12
    assert abs(cdf[0] - 0.12966) < 5e-5           # rank-1 share
    assert abs(cdf[9] - 0.3475) < 5e-4            # top-10 mass
    assert abs(cdf[999] - 0.7226) < 5e-4          # top-1000 mass
    assert np.array_equal(np.sort(perm), np.arange(num_bins, dtype=np.uint32))
    keys = gen.zipf(1 << 21, num_bins, seed=0, s=s)
    h1 = np.bincount(keys, minlength=num_bins)
    assert h1.argmax() == perm[0]
    assert abs(h1.max() / keys.size - 1 / h) < 0.002


def test_runs_structure():
    n, num_bins, run = 1 << 16, 512, 256
    keys = gen.runs(n, num_bins, seed=3, run_len=run)
    tail = keys[n // 2:].reshape(-1, run)
    assert (tail == tail[:, :1]).all()
    assert keys.min() >= 0 and keys.max() < num_bins
    assert len(np.unique(tail[:, 0])) > 50


def test_hot_generator_share_and_bin():
    n, num_bins = 1 << 20, 262144
    keys = gen.hot(n, num_bins, seed=5, share=0.25)
    hb = gen.hot_bin(num_bins, 5)
    counts = np.bincount(keys, minlength=num_bins)
    assert counts.argmax() == hb
    # a quarter of the keys are the hot bin (binomial sd about 0.0004 here),
    # plus its ordinary uniform share
    assert abs(counts[hb] / n - (0.25 + 0.75 / num_bins)) < 0.003
    assert keys.min() >= 0 and keys.max() < num_bins
    # the same bytes whatever the thread count
    assert np.array_equal(keys, gen.hot(n, num_bins, seed=5, share=0.25, threads=1))
    assert np.array_equal(gen.workload("hot25-256M-256K", 5, n=n), keys)
