"""Failure detection on the GPU, in forms that fault, trap or hang nothing.

- A bounded inbox wait of the key-shipping kernel runs out: the senders of a
  test launch withhold their last round's arrival and stores (so nothing is
  in flight), and the wait bound is cut to 2e5 cycles.  The launch returns
  normally, its histogram is short, the next call on the same stream reports
  DSMEM_HIST_ETIMEOUT without enqueueing anything, a call on another stream
  is unaffected, the device-wide word reads ETIMEOUT once, and the next
  normal call is bit-exact against the oracle.
- The scratch allocation fails (injected on the host): DSMEM_HIST_ENOMEM, and
  the library stays usable.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import cluster_distributed_shared_gb300 as pkg  # noqa: E402
import gen  # noqa: E402
import oracle  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    yield
    torch.cuda.synchronize()


def _call(fn, keys, num_bins, out, stream):
    return getattr(pkg.lib(), fn)(ctypes.c_void_p(keys.data_ptr()), keys.numel(), num_bins,
                                  ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(stream.cuda_stream))


def _bits(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("fn", ["dsmem_hist", "dsmem_hist_static"])
def test_inbox_wait_runs_out_and_the_next_call_reports_it(monkeypatch, fn):
    num_bins, n = 262144, 1 << 23          # P = 8, several rounds per CTA
    keys_np = gen.uniform(n, num_bins, seed=71)
    keys = torch.from_numpy(keys_np).cuda()
    want = oracle.histogram(keys_np, num_bins)
    s, other = torch.cuda.Stream(), torch.cuda.Stream()
    out = torch.zeros(num_bins, dtype=torch.int32, device="cuda")
    # make sure this stream's host-mapped word exists (dsmem_hist_static
    # allocates nothing itself)
    assert _call("dsmem_hist", keys, num_bins, out, s) == pkg.DSMEM_HIST_OK
    s.synchronize()
    assert pkg.dsmem_hist_plan(num_bins, n)["kernel"] == pkg.KERNEL_SHIP

    monkeypatch.setenv("DSMEM_HIST_TEST_WITHHOLD_LAST_ROUND", "1")
    monkeypatch.setenv("DSMEM_HIST_TEST_WAIT_CYCLES", "200000")
    assert _call(fn, keys, num_bins, out, s) == pkg.DSMEM_HIST_OK   # the launch itself is fine
    s.synchronize()
    monkeypatch.delenv("DSMEM_HIST_TEST_WITHHOLD_LAST_ROUND")
    monkeypatch.delenv("DSMEM_HIST_TEST_WAIT_CYCLES")
    short = _bits(out)
    assert int(short.sum(dtype=np.uint64)) < n    # the withheld round's keys never arrived
    assert not np.array_equal(short, want)

    # Another stream has its own word: unaffected.
    out2 = torch.zeros(num_bins, dtype=torch.int32, device="cuda")
    assert _call(fn, keys, num_bins, out2, other) == pkg.DSMEM_HIST_OK
    other.synchronize()
    assert np.array_equal(_bits(out2), want)

    # The same stream: the next call reports the timeout once and enqueues nothing.
    sentinel = torch.full((num_bins,), 7, dtype=torch.int32, device="cuda")
    assert _call(fn, keys, num_bins, sentinel, s) == pkg.DSMEM_HIST_ETIMEOUT
    assert b"wait give up" in pkg.lib().dsmem_hist_last_error()
    s.synchronize()
    assert (sentinel == 7).all().item()
    assert _call(fn, keys, num_bins, out, s) == pkg.DSMEM_HIST_OK
    s.synchronize()
    assert np.array_equal(_bits(out), want)

    # The device-wide word saw it too, and reads clear afterwards.
    torch.cuda.synchronize()
    assert pkg.dsmem_hist_device_status() == 1
    assert pkg.dsmem_hist_device_status() == 0


def test_partials_entry_reports_a_timeout_of_an_earlier_launch(monkeypatch):
    num_bins, n = 65536, 1 << 22             # P = 2
    keys_np = gen.uniform(n, num_bins, seed=72)
    keys = torch.from_numpy(keys_np).cuda()
    plan = pkg.dsmem_hist_plan(num_bins, n, cluster_size=2, kernel=pkg.KERNEL_SHIP)
    partials = torch.empty(-(-plan["workspace_bytes"] // 4), dtype=torch.int32,
                           device="cuda")
    s = torch.cuda.Stream()
    monkeypatch.setenv("DSMEM_HIST_TEST_WITHHOLD_LAST_ROUND", "1")
    monkeypatch.setenv("DSMEM_HIST_TEST_WAIT_CYCLES", "100000")
    pkg.dsmem_hist_partials(keys, num_bins, plan, partials, 0, s)
    s.synchronize()
    monkeypatch.delenv("DSMEM_HIST_TEST_WITHHOLD_LAST_ROUND")
    monkeypatch.delenv("DSMEM_HIST_TEST_WAIT_CYCLES")
    with pytest.raises(pkg.DsmemHistError) as e:
        pkg.dsmem_hist_partials(keys, num_bins, plan, partials, 0, s)
    assert e.value.code == pkg.DSMEM_HIST_ETIMEOUT
    pkg.dsmem_hist_partials(keys, num_bins, plan, partials, 0, s)
    bins = pkg.dsmem_hist_reduce(partials, plan["partial_rows"], plan["partial_stride"],
                                 num_bins, stream=s)
    s.synchronize()
    assert np.array_equal(_bits(bins), oracle.histogram(keys_np, num_bins))
    torch.cuda.synchronize()
    assert pkg.dsmem_hist_device_status() == 1


def test_injected_scratch_failure_returns_enomem_and_library_stays_usable(monkeypatch):
    num_bins = 262144
    keys_np = gen.uniform(1 << 22, num_bins, seed=73)
    keys = torch.from_numpy(keys_np).cuda()
    want = oracle.histogram(keys_np, num_bins)
    out = torch.full((num_bins,), 5, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream()
    monkeypatch.setenv("DSMEM_HIST_TEST_FAIL_ALLOC", "1")
    assert _call("dsmem_hist", keys, num_bins, out, s) == pkg.DSMEM_HIST_ENOMEM
    assert b"DSMEM_HIST_TEST_FAIL_ALLOC" in pkg.lib().dsmem_hist_last_error()
    with pytest.raises(pkg.DsmemHistError) as e:
        pkg.dsmem_hist_host(keys_np, num_bins)
    assert e.value.code == pkg.DSMEM_HIST_ENOMEM
    with pytest.raises(pkg.DsmemHistError) as e:
        pkg.dsmem_hist_tune(keys, num_bins, sample_keys=1 << 20)
    assert e.value.code == pkg.DSMEM_HIST_ENOMEM
    # the allocation-free entry point does not allocate, so it is unaffected
    assert _call("dsmem_hist_static", keys, num_bins, out, s) == pkg.DSMEM_HIST_OK
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), want)
    monkeypatch.delenv("DSMEM_HIST_TEST_FAIL_ALLOC")
    out.fill_(5)
    assert _call("dsmem_hist", keys, num_bins, out, s) == pkg.DSMEM_HIST_OK
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), want)
    assert np.array_equal(pkg.dsmem_hist_host(keys_np, num_bins), want)
