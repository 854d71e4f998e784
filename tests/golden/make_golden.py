"""Write the golden regression fixtures in this folder.

Calls only the seeded generators (gen/) and the CPU oracle (oracle/): the
stored digests pin the generators' bytes and the oracle's counts across hosts
(x86_64 and aarch64 must agree).  The counts follow the histogram definition
of "Distributed Shared Memory", section "The cluster histogram".

Run from the repository root:  python tests/golden/make_golden.py
"""
from __future__ import annotations

import hashlib
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import gen  # noqa: E402
import oracle  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def digest(a):
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def write(name, keys, num_bins, meta):
    bins = oracle.histogram(keys, num_bins)
    top = np.argsort(-bins.astype(np.int64), kind="stable")[:4]
    sample = [[int(b), int(bins[b])] for b in [0, num_bins // 2, num_bins - 1, *top]]
    rec = dict(meta, num_bins=num_bins, sha256_keys=digest(keys), sha256_bins=digest(bins),
               in_range=int(bins.sum(dtype=np.uint64)), sample=sample,
               source="tests/golden/make_golden.py (gen + oracle); definition: "
                      "'Distributed Shared Memory', section 'The cluster histogram'")
    with open(os.path.join(HERE, name), "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")


def main():
    write("uniform-1M-8K_seed0.json", gen.workload("uniform-1M-8K", 0), 8192,
          dict(workload="uniform-1M-8K", seed=0))
    write("runs256-64K-512_seed3.json", gen.runs(65536, 512, 3, 256), 512,
          dict(dist="runs", args=dict(n=65536, num_bins=512, seed=3, run_len=256)))
    write("uniform-nonpow2-100003-1000_seed9.json", gen.uniform(100003, 1000, 9), 1000,
          dict(dist="uniform", args=dict(n=100003, num_bins=1000, seed=9)))


if __name__ == "__main__":
    main()
