"""The benchmark's multi-rank host logic on CPU (gloo, world size 2): the
path shards into independent replicas, so the only cross-rank work is the
barrier, the max over ranks of the timed region and the sum of the work."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import bench
    w, r, _ = bench.dist_info()
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    mx = bench.max_over_ranks(10.0 + r, w)
    sm = bench.sum_over_ranks(1.5 * (r + 1), w)
    ref = bench.reference_arm(type("A", (), dict(steps=1, warmup=0,
                                                 ref_seconds=0.0))(), w, r) \
        if r != 0 else "skip"
    q.put((r, mx, sm, ref))
    torch.distributed.destroy_process_group()


def test_two_ranks_max_and_sum():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, mx, sm, ref in res:
        assert mx == 11.0
        assert sm == pytest.approx(1.5 + 3.0)
        if r == 1:
            assert ref is None     # only rank 0 runs and prints the reference arm
