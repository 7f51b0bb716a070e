"""bench.py's multi-rank path on CPU: two gloo ranks (no GPU).

Under torchrun every rank runs its own copy of the workload; the timed region
is bracketed by barriers and the reported time is the maximum over ranks; the
reference (oracle) arm runs on rank 0 only and the other ranks exit without
work. These are checked with world_size 2 on the gloo backend.
"""
import argparse
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      VA_BENCH_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    t = bench.max_over_ranks(1.5 + r, w, None)        # rank-dependent "time"
    bench.barrier(w)
    args = argparse.Namespace(steps=1, warmup=3, reference_rows=2, workload="wan_radial")
    line = bench.run_reference(args, w, r)
    out.put((r, w, t, None if line is None else (line["impl"], line["n_gpus"],
                                                  line["cpu_baseline"]["kind"])))
    dist.destroy_process_group()


@pytest.mark.slow
def test_two_gloo_ranks_max_time_and_rank0_reference():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1] and all(x[1] == 2 for x in res)
    assert all(x[2] == 2.5 for x in res)                # max over the two ranks
    assert res[0][3] == ("reference", 1, "oracle")      # rank 0 runs the oracle arm
    assert res[1][3] is None                            # rank 1 exits without work
