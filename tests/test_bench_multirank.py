"""Host logic of bench.py's multi-rank path, on CPU with gloo (world size 2).

Under torchrun every rank histograms its own replica (weak scaling, no
collective on the data path); the reported time is the slowest rank's and
the rate counts every rank's keys.  The reference arm runs on rank 0 only.
"""
from __future__ import annotations

import io
import os
import socket
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]
        results[rank] = (bench.max_over_ranks(local_ms, dist), bench.replica_seed(7, rank))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_replica_seeds_gloo():
    world, port = 2, _free_port()
    manager = mp.Manager()
    results = manager.dict()
    mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
    assert results[0][0] == results[1][0] == 5.0      # slowest rank's time everywhere
    assert results[0][1] != results[1][1]              # independent replicas


def test_whole_job_rate_counts_every_rank():
    assert bench.whole_job_rate(1, 1000, 10, 1.0) == pytest.approx(1e7)
    assert bench.whole_job_rate(4, 1000, 10, 1.0) == pytest.approx(4e7)
    assert bench.max_over_ranks(2.5) == 2.5


def test_reference_arm_runs_on_rank_zero_only():
    class A:
        workload, seed, steps, warmup, keys = "uniform-1M-8K", 0, 5, 3, 0
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(A, world=2, rank=1)
    assert buf.getvalue() == ""
    with redirect_stdout(buf):
        bench.run_reference(A, world=2, rank=0)
    import json
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_keys_override_scales_a_workload():
    import numpy as np
    import gen
    cfg = bench.workload_config("runs256-1G-512K", 0, 1 << 20)
    assert cfg["n"] == 1 << 20 and cfg["num_bins"] == 524288 and cfg["keys_override"]
    assert "keys_override" not in bench.workload_config("runs256-1G-512K", 0)
    k = gen.workload("runs256-1G-512K", 3, n=1 << 12)
    assert k.size == 1 << 12
    # Same layout as the full workload: uniform first half, runs of 256 after it.
    runs = k[2048:].reshape(-1, 256)
    assert (runs == runs[:, :1]).all() and runs.shape == (8, 256)
    assert np.unique(k[:2048]).size > 1000
