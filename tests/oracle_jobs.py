"""Per-head oracle jobs for a spawn process pool (full-size GPU parity tests).

Each job takes picklable arrays, calls only the float64 oracle, and returns
small numpy results, so the heads of a full-size workload can be checked side
by side. The pool is started with the spawn method: its workers never touch
CUDA and do not inherit the test process's CUDA context.
"""
from __future__ import annotations

import multiprocessing
import os

import numpy as np

from oracle import kmeans as KM
from oracle import svgear as S


def lloyd_run(x, init_idx, iters):
    """The oracle's own Lloyd run: (assign, inertia)."""
    a, c, _ = KM.lloyd(x, init_idx, iters)
    return a, KM.inertia(x, a, c)


def probe_err(q, k, v, qa, Cq, ka, Ck, scale):
    """The oracle's float64 probe errors err [Cq, Ck] on the given clusters."""
    return S.probe(q, k, v, qa, Cq, ka, Ck, scale)["err"]


def spawn_pool(jobs: int):
    """A spawn-method pool of single-threaded workers (BLAS threads = 1)."""
    n = max(1, min(jobs, os.cpu_count() or 1))
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = "1"
    try:
        return multiprocessing.get_context("spawn").Pool(n)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
