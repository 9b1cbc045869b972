"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2): the
barrier + max-over-ranks timing and the whole-job weak-scaling throughput, and
that ranks serve disjoint synthetic streams."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, local, w = bench.dist_init("gloo")
    bench.barrier()
    ms_local = 10.0 + 5.0 * rank                      # rank 1 is the slow one
    value, ms_max = bench.aggregate_throughput(ms_local, streams=256, frames=2, steps=100, device=torch.device("cpu"))
    from cache_aware_conformer_gb300 import synth
    offs = synth.start_offsets(8, 500, seed=7 + rank)
    q.put((r, w, value, ms_max, offs.tolist()))
    dist.destroy_process_group()


def test_two_ranks_gloo_max_time_and_weak_scaling():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, v0, m0, o0), (r1, w1, v1, m1, o1) = out
    assert (r0, r1, w0, w1) == (0, 1, 2, 2)
    assert m0 == m1 == 15.0                          # max over ranks, seen by every rank
    expect = 2 * 256 * 2 * 0.08 * 100 / 0.015       # both ranks' audio over the slowest rank's time
    assert np.isclose(v0, expect) and np.isclose(v1, expect)
    assert o0 != o1                                  # ranks draw different start offsets
