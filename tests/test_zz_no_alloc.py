"""The allocation-free entry point, dsmem_hist_static, against the CPU oracle
and against dsmem_hist.

Callers that cannot let a library allocate device memory (code running
under stream capture, applications that own every byte through their own
arena, allocator-free hot paths) call dsmem_hist_static, which keeps its
partial histograms in a fixed 32 MiB static device array.  Every result here
is compared bit for bit with the oracle; the comparison with dsmem_hist is a
second check.  This file is named so that pytest collects it last: if it
fails, a run that stops at the first failure has already run every other
test.
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

STATIC_BYTES = 32 << 20       # the library's static scratch
MAX_BINS = STATIC_BYTES // 4  # 8,388,608


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    yield
    torch.cuda.synchronize()


def _static_via_c_abi(keys, num_bins, out=None, stream=None):
    if out is None:
        out = torch.full((num_bins,), -1, dtype=torch.int32, device=keys.device)
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = pkg.lib().dsmem_hist_static(ctypes.c_void_p(keys.data_ptr()), keys.numel(), num_bins,
                                     ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(s.cuda_stream))
    assert rc == pkg.DSMEM_HIST_OK, pkg.lib().dsmem_hist_last_error()
    return out


def _bits(t):
    return t.cpu().numpy().view(np.uint32)


def _static_clusters(num_bins, n):
    """Clusters the static path launches: the planner's count, cut to the
    partial rows that fit the static scratch."""
    plan = pkg.dsmem_hist_plan(num_bins, n)
    row_bytes = 4 * ((num_bins + 3) // 4 * 4)
    return plan, min(plan["num_clusters"], STATIC_BYTES // row_bytes)


def test_static_matches_oracle_and_dsmem_hist_on_two_calls_in_a_row():
    inputs = [
        (gen.uniform(1 << 24, 262144, seed=31), 262144),
        (gen.zipf(1 << 23, 65536, seed=32), 65536),
    ]
    for keys_np, num_bins in inputs:  # two calls in a row on the shared static scratch
        keys = torch.from_numpy(keys_np).cuda()
        got = _static_via_c_abi(keys, num_bins)
        want = pkg.dsmem_hist(keys, num_bins)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(_bits(got), oracle.histogram(keys_np, num_bins))
        np.testing.assert_array_equal(_bits(got), _bits(want))  # integer counts: bit-exact


def test_static_with_many_bins_uses_fewer_clusters_and_rejects_too_many():
    n, num_bins = 1 << 22, 1 << 22
    keys_np = gen.uniform(n, num_bins, seed=33)
    keys = torch.from_numpy(keys_np).cuda()
    plan, clusters = _static_clusters(num_bins, n)
    # 4,194,304 bins: clusters of 16 x 32,768 counters in 8 passes; 16 MiB
    # partial rows, so the 32 MiB scratch holds 2 of them.
    assert plan["cluster_size"] == 16 and plan["bins_per_cta"] == 32768 and plan["passes"] == 8
    assert clusters == 2 < plan["num_clusters"]
    assert clusters * plan["partial_stride"] * 4 <= STATIC_BYTES
    got = _static_via_c_abi(keys, num_bins)
    want = pkg.dsmem_hist(keys, num_bins)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(got), oracle.histogram(keys_np, num_bins))
    np.testing.assert_array_equal(_bits(got), _bits(want))
    out = torch.empty(MAX_BINS + 1, dtype=torch.int32, device="cuda")
    rc = pkg.lib().dsmem_hist_static(ctypes.c_void_p(keys.data_ptr()), keys.numel(), MAX_BINS + 1,
                                     ctypes.c_void_p(out.data_ptr()), None)
    assert rc == pkg.DSMEM_HIST_EINVAL
    assert b"static scratch" in pkg.lib().dsmem_hist_last_error()


def test_static_at_the_largest_accepted_bin_count():
    # 8,388,608 bins: one 32 MiB partial row fills the scratch, so one
    # cluster of 16 CTAs streams the keys in 16 passes.
    n = 1 << 20
    keys_np = gen.uniform(n, MAX_BINS, seed=34)
    keys_np[:4096] = MAX_BINS - 1 - np.arange(4096, dtype=np.int32)  # the top bins too
    keys = torch.from_numpy(keys_np).cuda()
    plan, clusters = _static_clusters(MAX_BINS, n)
    assert plan["passes"] == 16 and clusters == 1
    got = _static_via_c_abi(keys, MAX_BINS)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(got), oracle.histogram(keys_np, MAX_BINS))


def test_static_call_captured_in_a_cuda_graph_replays_exactly():
    n, num_bins = 1 << 20, 65536
    keys_np = gen.uniform(n, num_bins, seed=35)
    keys = torch.from_numpy(keys_np).cuda()
    out = torch.zeros(num_bins, dtype=torch.int32, device="cuda")
    _static_via_c_abi(keys, num_bins, out)  # warm-up: device set-up and plan before capture
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            _static_via_c_abi(keys, num_bins, out, stream=side)
    torch.cuda.synchronize()
    out.fill_(-1)
    graph.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(out), oracle.histogram(keys_np, num_bins))
    keys_np2 = gen.zipf(n, num_bins, seed=36)   # new key contents in the captured buffer
    keys.copy_(torch.from_numpy(keys_np2))
    out.fill_(-1)
    graph.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(out), oracle.histogram(keys_np2, num_bins))
