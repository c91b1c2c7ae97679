"""Multi-rank host logic of bench.py on CPU: two gloo ranks.

Every rank runs its own independent projections (replicas, no data-path
collective); the only cross-rank step is the timing reduction: the elapsed
time is the maximum over ranks and the work done is the sum.  Run here as two
spawned processes on the gloo backend.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp

from tests.conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        ms = [12.5, 40.0][rank]
        units = [1000.0, 3000.0][rank]
        t, u = bench.aggregate(ms, units, dist)
        q.put((rank, (r, w, local), t, u))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction_is_max_time_and_summed_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    for rank, env, t, u in out:
        assert env == (rank, 2, rank)
        assert t == pytest.approx(40.0)      # the slowest rank sets the time
        assert u == pytest.approx(4000.0)    # units of every rank count


def test_single_rank_aggregate_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(3.0, 7.0, None) == (3.0, 7.0)
