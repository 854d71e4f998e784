"""GPU tests of the cluster-shape screen (dsmem_hist_tune) and the DSMEM
microbenchmarks (dsmem_hist_microbench)."""
from __future__ import annotations

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


@pytest.mark.parametrize("num_bins", [8192, 262144])
def test_tune_ranks_every_shape_and_its_winner_is_exact(num_bins):
    keys_np = gen.uniform(1 << 22, num_bins, seed=41)
    keys = torch.from_numpy(keys_np).cuda()
    res = pkg.dsmem_hist_tune(keys, num_bins, sample_keys=1 << 21)
    assert len(res) >= 3
    assert [r["ms"] for r in res] == sorted(r["ms"] for r in res)
    assert sum(r["global_atomic"] for r in res) == 1
    clustered = [r for r in res if not r["global_atomic"]]
    assert {r["cluster_size"] for r in clustered} >= {2, 8, 16}
    assert all(r["ms"] > 0 and r["control_ms"] > 0 for r in clustered)
    want = oracle.histogram(keys_np, num_bins)
    for r in clustered[:3]:  # the fastest shapes reproduce the exact histogram
        got = pkg.dsmem_hist(keys, num_bins, cluster_size=r["cluster_size"], kernel=r["kernel"],
                             block_threads=r["block_threads"], aggregate=r["aggregate"])
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy().view(np.uint32), want), r


def test_microbench_rates_are_consistent_and_did_their_counted_work():
    kinds = [k for k in pkg.MICROBENCH_KINDS if not k.startswith("tile_exchange")]
    rates = {k: pkg.dsmem_hist_microbench(k, 2, iters=512) for k in kinds}
    for k, r in rates.items():
        # every probe did exactly the work it claims: increments landed,
        # stores and barriers issued, round trips completed
        assert r["ops_counted"] == r["ops_expected"] > 0, r
        assert r["value"] > 0 and r["ms"] > 0, r
    assert rates["dsmem_pingpong"]["ops_expected"] == 512
    # one-way flag latency: hundreds to thousands of cycles, and a flag in a
    # peer's shared memory arrives no later than one in global memory
    for k in ("dsmem_pingpong", "gmem_pingpong"):
        assert 20 < rates[k]["value"] < 1e5, rates[k]
    assert rates["dsmem_pingpong"]["value"] < 1.5 * rates["gmem_pingpong"]["value"]
    # a local shared-memory atomic is far cheaper than a remote one
    assert rates["local_red"]["value"] > 4 * rates["remote_red"]["value"]
    # one cluster barrier costs at least tens of cycles and well under a million
    assert 10 < rates["cluster_barrier"]["value"] < 1e6
    # the same counts hold at the other cluster sizes the histogram uses
    for P in (1, 8, 16):
        for k in ("local_red", "remote_red", "remote_st16_coalesced", "cluster_barrier"):
            r = pkg.dsmem_hist_microbench(k, P, iters=64)
            assert r["ops_counted"] == r["ops_expected"] > 0, r
    import ctypes
    res = pkg.MicrobenchResult()
    assert pkg.lib().dsmem_hist_microbench(99, 2, 16, ctypes.byref(res)) == pkg.DSMEM_HIST_EINVAL


@pytest.mark.parametrize("P", [2, 4])
def test_tile_exchange_pair_moves_every_tile(P):
    iters = 500
    d = pkg.dsmem_hist_microbench("tile_exchange_dsmem", P, iters=iters)
    g = pkg.dsmem_hist_microbench("tile_exchange_gmem", P, iters=iters)
    for r in (d, g):
        # every word of the peer's tile arrived on every iteration
        assert r["ops_counted"] == r["ops_expected"] > 0, r
        assert r["ctas"] >= 2 * P and r["ctas"] % P == 0
        assert r["value"] == r["ms"] > 0
        assert r["bytes_per_s"] == pytest.approx(r["ctas"] * 16384 * iters / (r["ms"] * 1e-3))
    assert d["ctas"] == g["ctas"]
