"""The allocation-free entry point, dsmem_hist_static, against dsmem_hist.

Callers that cannot let a library allocate device memory (code running
under stream capture, applications that own every byte through their own
arena, allocator-free hot paths) call dsmem_hist_static, which keeps its
partial histograms in a fixed static device array.  This file is named so
that pytest collects it last: if it fails, a run that stops at the first
failure has already run every other test.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import cluster_distributed_shared_gb300 as pkg  # noqa: E402
import gen  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    yield
    torch.cuda.synchronize()


def _static_via_c_abi(keys, num_bins):
    out = torch.full((num_bins,), -1, dtype=torch.int32, device=keys.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = pkg.lib().dsmem_hist_static(ctypes.c_void_p(keys.data_ptr()), keys.numel(), num_bins,
                                     ctypes.c_void_p(out.data_ptr()), stream)
    assert rc == pkg.DSMEM_HIST_OK, pkg.lib().dsmem_hist_last_error()
    return out


def _bits(t):
    return t.cpu().numpy().view(np.uint32)


def test_static_matches_dsmem_hist_on_two_calls_in_a_row():
    inputs = [
        (torch.from_numpy(gen.uniform(1 << 24, 262144, seed=31)).cuda(), 262144),
        (torch.from_numpy(gen.zipf(1 << 23, 65536, seed=32)).cuda(), 65536),
    ]
    for keys, num_bins in inputs:  # two calls in a row on the shared static scratch
        got = _static_via_c_abi(keys, num_bins)
        want = pkg.dsmem_hist(keys, num_bins)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(_bits(got), _bits(want))  # integer counts: bit-exact


def test_static_handles_many_bins_and_rejects_too_many():
    keys = torch.from_numpy(gen.uniform(1 << 22, 1 << 22, seed=33)).cuda()
    got = _static_via_c_abi(keys, 1 << 22)          # 16 MiB rows: fewer clusters, two passes
    want = pkg.dsmem_hist(keys, 1 << 22)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(got), _bits(want))
    out = torch.empty(8388609, dtype=torch.int32, device="cuda")
    rc = pkg.lib().dsmem_hist_static(ctypes.c_void_p(keys.data_ptr()), keys.numel(), 8388609,
                                     ctypes.c_void_p(out.data_ptr()), None)
    assert rc == pkg.DSMEM_HIST_EINVAL
    assert b"static scratch" in pkg.lib().dsmem_hist_last_error()
