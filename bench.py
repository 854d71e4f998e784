"""Benchmark of the thread-block-cluster histogram on one GB300 (or N replicas).

One step = one whole histogram of the workload's keys: the cluster kernel
(zero slices, stream keys, DSMEM increments, flush partial rows) followed by
the partial-row reduction, both launched through the library's C ABI.  Keys
are resident in HBM when the timed region starts; the 1 GiB input is larger
than the 129 MB L2, so no flush is needed between steps.

Prints ONE JSON line on rank 0.  Under torchrun (N > 1) every rank runs an
independent replica on its own GPU with its own seed (weak scaling; there is
no collective on the data path) and the slowest rank's time is reported.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle as the reference arm
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "keys/s and achieved HBM GB/s vs GB300 peak (1 GPU), bit-exact vs CPU oracle"
UNIT = "keys/s"
DEFAULT_WORKLOAD = "uniform-256M-256K"
# Cluster size each synthetic workload is published with.
WORKLOAD_CLUSTER = {
    "uniform-1M-8K": 2,
    "uniform-64M-64K": 2,
    "uniform-256M-256K": 8,
    "zipf1.1-256M-256K": 8,
    "runs256-1G-512K": 16,
    "hot25-256M-256K": 8,   # skewed case: a quarter of the keys on one bin
}
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 1024 * 1024
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "cluster_hist_traffic.json")
KERNEL_SOURCES = {  # plan kernel id -> (kernel name, source file)
    0: ("cluster_hist_kernel", os.path.join(ROOT, "cluster_distributed_shared_gb300", "csrc",
                                            "cluster_hist.cu")),
    1: ("cluster_ship_kernel", os.path.join(ROOT, "cluster_distributed_shared_gb300", "csrc",
                                            "cluster_ship.cu")),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOAD_CLUSTER))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--keys", type=int, default=0,
                    help="scale the workload to this many keys, same distribution (profiling of "
                         "smaller cases; default: the workload's own length)")
    ap.add_argument("--cluster", type=int, default=0,
                    help="cluster size (default: the workload's published one)")
    ap.add_argument("--hot-bin-hint", action="store_true",
                    help="hot25 workload: tell the library its hot bin (the hinted ship kernel)")
    a = ap.parse_args()
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    if a.steps < 1:
        ap.error("--steps must be >= 1")
    if a.keys < 0 or (a.keys and a.keys % 512):
        ap.error("--keys must be a positive multiple of 512 (whole runs of 256 in either half)")
    return a


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def workload_config(name, seed, keys=0):
    """The named workload's description; `keys` > 0 scales it to that many keys
    (same distribution; a profiling aid, reported in the config)."""
    import gen
    w = dict(gen.WORKLOADS[name])
    if keys:
        w["n"] = keys
    return {
        "workload": name,
        "n": w["n"],
        "num_bins": w["num_bins"],
        "distribution": w["dist"],
        "seed": seed,
        "cluster_size": WORKLOAD_CLUSTER[name],
        "l2": "inputs larger than L2 (no flush)" if 4 * w["n"] > L2_BYTES
        else "inputs L2-resident (smaller than L2; no flush)",
        **({"keys_override": True} if keys else {}),
    }


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [l for (t, l) in self.lines if t0 - 0.06 <= t <= t1 + 0.06] or \
               [l for (_, l) in self.lines]
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {
            "sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "power_w_max": max(power) if power else None,
            "samples": len(sm),
            "reasons": sorted(reasons),
        }


def gpu_id_for(torch, dev_index):
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[dev_index] if vis else str(dev_index)


# ---------------------------------------------------------------- peaks

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# Files whose bytes decide the compiled cluster kernels: a change to any of
# them invalidates the committed DRAM counters.
KERNEL_DEPENDENCIES = [
    os.path.join(ROOT, "cluster_distributed_shared_gb300", "csrc", "ptx.cuh"),
    os.path.join(ROOT, "cluster_distributed_shared_gb300", "csrc", "internal.h"),
    os.path.join(ROOT, "include", "dsmem_hist.h"),
]


def kernel_sources_sha256(kernel_id):
    """sha256 over the kernel's source file and the headers it includes."""
    h = hashlib.sha256()
    for path in [KERNEL_SOURCES[kernel_id][1]] + KERNEL_DEPENDENCIES:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def kernel_traffic(workload, n_keys, num_bins, cluster_size, kernel_id, block_threads):
    """DRAM bytes of one partials stage (the cluster kernel, plus the idle-SM
    helper where the capture has one) from the committed ncu summary of the
    same workload, scaled to this launch's keys; None when no capture of that
    workload and shape exists or the kernels' sources or the block size have
    changed since the counters were taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
        name = KERNEL_SOURCES[kernel_id][0]
        sha = kernel_sources_sha256(kernel_id)
        if not rec.get("kernel", "").startswith(name):
            return None
    except (OSError, ValueError, KeyError):
        return None
    if rec.get("kernel_sources_sha256") != sha:
        return None
    for e in rec.get("captures", []):
        if (e.get("workload") == workload and e.get("num_bins") == num_bins
                and e.get("cluster_size") == cluster_size and e.get("block_threads") == block_threads):
            return e["dram_bytes"] * (n_keys / e["n"])
    return None


ARM_PARTS = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1", "0xd49": "Arm Neoverse N2",
             "0xd0c": "Arm Neoverse N1"}


def host_info():
    """The host the CPU baseline ran on: logical CPUs and the CPU model."""
    model = platform.processor() or platform.machine()
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip().lower(), v.strip())
    except OSError:
        pass
    if "model name" in fields:
        model = fields["model name"]
    elif "cpu part" in fields:
        part = fields["cpu part"].lower()
        model = ARM_PARTS.get(part, f"Arm CPU part {part}") + f" ({platform.machine()})"
    return {"host_cpus": os.cpu_count(), "cpu_model": model}


# ---------------------------------------------------------------- multi-rank

def replica_seed(seed, rank):
    """Each rank histograms its own independent replica of the workload."""
    return seed + rank


def max_over_ranks(x, dist=None, device=None):
    """The slowest rank's value (time), via one MAX all-reduce; the rank's
    own value when running alone."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, n, steps, ms_total):
    """Keys per second over all ranks: every rank processed n keys per step."""
    return world * n * steps / (ms_total / 1e3)


# ---------------------------------------------------------------- reference arm

def run_reference(a, world, rank):
    if rank != 0:
        return
    import gen
    import oracle
    cfg = workload_config(a.workload, a.seed, a.keys)
    keys = gen.workload(a.workload, a.seed, n=cfg["n"])
    n, num_bins = cfg["n"], cfg["num_bins"]
    # Size each step's sample so the whole run stays around a minute.
    probe = keys[: 1 << 20]
    t0 = time.perf_counter()
    oracle.histogram(probe, num_bins)
    t_key = max((time.perf_counter() - t0) / probe.size, 1e-10)
    sample = int(min(n, max(1 << 16, 40.0 / ((a.steps + a.warmup) * t_key))))
    sample = max(sample - sample % 4096, 4096)
    out = np.empty(num_bins, np.uint32)
    chunks = max(1, n // sample)
    for k in range(a.warmup):
        o = (k % chunks) * sample
        oracle.histogram(keys[o:o + sample], num_bins, out)
    t0 = time.perf_counter()
    for k in range(a.steps):
        o = (k % chunks) * sample
        oracle.histogram(keys[o:o + sample], num_bins, out)
    dt = time.perf_counter() - t0
    value = sample * a.steps / dt
    desc = (f"{sample} contiguous keys of the {n}-key workload per step, cycling through it; "
            "single-threaded C loop")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1e3 * dt / a.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic (seeded generator)", "config": cfg,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": desc, **host_info()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm

def run_ours(a, world, rank, local):
    import torch
    import cluster_distributed_shared_gb300 as pkg
    import gen

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    cfg = workload_config(a.workload, a.seed, a.keys)
    seed = replica_seed(a.seed, rank)
    if a.cluster:
        cfg["cluster_size"] = a.cluster
    n, num_bins, P = cfg["n"], cfg["num_bins"], cfg["cluster_size"]
    keys_h = gen.workload(a.workload, seed, n=cfg["n"])
    keys = torch.from_numpy(keys_h).to(dev)
    hint = {}
    if a.hot_bin_hint:
        if gen.WORKLOADS[a.workload]["dist"] != "hot":
            raise SystemExit("--hot-bin-hint applies to the hot25 workload only")
        hint = {"hot_bin": gen.hot_bin(num_bins, seed)}
        cfg["hot_bin_hint"] = hint["hot_bin"]
    plan = pkg.dsmem_hist_plan(num_bins, n, cluster_size=P, **hint)
    partials = torch.empty(-(-plan["workspace_bytes"] // 4), dtype=torch.int32,
                           device=dev)
    bins = torch.empty(num_bins, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        pkg.dsmem_hist_partials(keys, num_bins, plan, partials, 0, stream)
        pkg.dsmem_hist_reduce(partials, plan["partial_rows"], plan["partial_stride"], num_bins,
                              bins, stream)

    # Warm-up steps wait for the GPU one by one, so that the library's
    # per-stream state (the helper's share, the hot-bin choice) settles on
    # reports of the steps just run rather than of steps long queued.
    for _ in range(a.warmup):
        step()
        torch.cuda.synchronize(dev)

    # Parity of the benchmarked configuration (rank 0 at N = 1 compares with
    # the oracle; the oracle run doubles as the CPU baseline).
    parity = None
    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        import oracle
        med, reps = oracle.time_histogram(keys_h, num_bins, min_seconds=a.cpu_seconds)
        want = oracle.histogram(keys_h, num_bins)
        got = bins.cpu().numpy().view(np.uint32)
        parity = "bit-exact vs oracle" if np.array_equal(got, want) else \
            f"MISMATCH in {int((got != want).sum())} bins"
        cpu = {"value": n / med, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"full {n}-key workload (seed {seed}), median of {reps} runs",
               **host_info()}

    sampler = ClockSampler(gpu_id_for(torch, local))
    sampler.start()
    ev_start = torch.cuda.Event(enable_timing=True)
    ev_end = torch.cuda.Event(enable_timing=True)
    ev_k = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(a.steps)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    t_host0 = time.perf_counter()
    ev_start.record(stream)
    for k in range(a.steps):
        ev_k[k][0].record(stream)
        pkg.dsmem_hist_partials(keys, num_bins, plan, partials, 0, stream)
        ev_k[k][1].record(stream)
        pkg.dsmem_hist_reduce(partials, plan["partial_rows"], plan["partial_stride"], num_bins,
                              bins, stream)
    ev_end.record(stream)
    torch.cuda.synchronize(dev)
    t_host1 = time.perf_counter()
    if pg:
        pg.barrier()
    clocks = sampler.stop(t_host0, t_host1)
    ms_total = ev_start.elapsed_time(ev_end)
    kernel_ms = [s.elapsed_time(e) for s, e in ev_k]
    cluster_ms = sum(kernel_ms) / len(kernel_ms)
    launch_stats = {"median": statistics.median(kernel_ms), "min": min(kernel_ms),
                    "max": max(kernel_ms)}
    if parity is not None:
        # The timed launches wrote `bins` too: check their result as well.
        got = bins.cpu().numpy().view(np.uint32)
        if not np.array_equal(got, want):
            parity = f"MISMATCH after the timed launches in {int((got != want).sum())} bins"
    ms_total = max_over_ranks(ms_total, pg, dev)
    ms_step = ms_total / a.steps
    value = whole_job_rate(world, n, a.steps, ms_total)

    # The product call dsmem_hist itself, timed the same way: it plans (from
    # the cache), takes its partial rows from the stream-ordered pool, launches
    # both kernels and returns the rows to the pool, every call.
    prod_steps = max(1, min(a.steps, 500))
    prod_out = torch.empty(num_bins, dtype=torch.int32, device=dev)
    for _ in range(max(3, a.warmup)):
        pkg.dsmem_hist(keys, num_bins, out=prod_out, stream=stream, **hint)
        torch.cuda.synchronize(dev)
    ev_start.record(stream)
    for _ in range(prod_steps):
        pkg.dsmem_hist(keys, num_bins, out=prod_out, stream=stream, **hint)
    ev_end.record(stream)
    torch.cuda.synchronize(dev)
    prod_ms = ev_start.elapsed_time(ev_end) / prod_steps
    product_call = {"call": "dsmem_hist (planner, pool scratch alloc + free, cluster kernel, "
                            "reduction)",
                    "plan": {k: v for k, v in pkg.dsmem_hist_plan(num_bins, n, **hint).items()
                             if k in ("cluster_size", "num_clusters", "kernel", "passes",
                                      "hot_bin")},
                    "ms_per_step": prod_ms, "value": world * n / (prod_ms / 1e3), "unit": UNIT,
                    "steps": prod_steps}
    if parity is not None:
        product_call["parity"] = ("bit-exact vs oracle" if np.array_equal(
            prod_out.cpu().numpy().view(np.uint32), want) else "MISMATCH")

    # The global-atomics comparison kernel, timed the same way on the same keys.
    cmp_steps = max(1, min(a.steps, 50))
    for _ in range(3):
        pkg.dsmem_hist_global_atomic(keys, num_bins, out=bins, stream=stream)
    torch.cuda.synchronize(dev)
    ev_start.record(stream)
    for _ in range(cmp_steps):
        pkg.dsmem_hist_global_atomic(keys, num_bins, out=bins, stream=stream)
    ev_end.record(stream)
    torch.cuda.synchronize(dev)
    ga_ms = ev_start.elapsed_time(ev_end) / cmp_steps
    comparison = {"kernel": "global_atomic_hist_kernel (one global atomic per key)",
                  "ms_per_step": ga_ms, "value": n / (ga_ms / 1e3), "unit": UNIT,
                  "steps": cmp_steps}

    # End to end through the host-buffer entry point: pinned keys in, the
    # histogram back in host memory, every step.
    e2e = None
    if not a.no_e2e:
        keys_pin = torch.from_numpy(keys_h).pin_memory()
        out_pin = torch.empty(num_bins, dtype=torch.int32).pin_memory()
        pkg.dsmem_hist_host(keys_pin, num_bins, out=out_pin)  # warm the staging pool
        e2e_steps = max(1, min(a.e2e_steps, a.steps))
        if pg:
            pg.barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            pkg.dsmem_hist_host(keys_pin, num_bins, out=out_pin)
        dt = max_over_ranks(time.perf_counter() - t0, pg, dev)
        ok = parity is None or np.array_equal(out_pin.numpy().view(np.uint32), want)
        e2e = {"value": world * n * e2e_steps / dt, "unit": UNIT,
               "h2d_bytes_per_step": 4 * n, "d2h_bytes_per_step": 4 * num_bins,
               "steps": e2e_steps, "call": "dsmem_hist_host (pinned host keys -> host bins)",
               "parity": "bit-exact vs oracle" if ok else "MISMATCH"}
        del keys_pin, out_pin

    peak, peak_src = hbm_peak()
    alg_bytes = 4 * n + 4 * num_bins
    achieved = alg_bytes / (cluster_ms / 1e3) / 1e9
    traffic = kernel_traffic(cfg["workload"], n, num_bins, P, plan["kernel"], plan["block_threads"])
    helper = plan["partial_rows"] > plan["num_clusters"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32", "data": "synthetic (seeded generator)",
        "config": cfg,
        "plan": plan,
        "achieved_gbs": world * alg_bytes / (ms_step / 1e3) / 1e9,
        "pct_of_nominal_8tbs": 100.0 * (alg_bytes / (ms_step / 1e3) / 1e9) / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "kernel": KERNEL_SOURCES[plan["kernel"]][0],
                     "stage": ("partials stage: the cluster kernel and, on the SMs its clusters "
                               "leave idle, the helper kernel (second stream, forked and joined), "
                               "then the mop-up kernel" if helper else
                               "partials stage: the cluster kernel"),
                     "achieved": achieved,
                     "peak": peak, "peak_source": peak_src, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes": alg_bytes, "avg_launch_ms": cluster_ms,
                     "launch_ms": launch_stats, "share_of_step": cluster_ms / ms_step},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "product_call": product_call,
        "global_atomic_comparison": comparison,
        # timed region, per step: the cluster kernel, the helper and the mop-up (if
        # planned), the reduction
        "gpu_launches": (4 if helper else 2) * a.steps,
        "clocks": clocks,
        "parity": parity,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


def main():
    a = parse()
    world, rank, local = dist_env()
    if a.impl == "reference":
        run_reference(a, world, rank)
    else:
        run_ours(a, world, rank, local)


if __name__ == "__main__":
    main()
