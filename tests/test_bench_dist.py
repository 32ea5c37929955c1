"""Host-side logic of the multi-GPU bench path, on CPU with gloo (world size 2).

The data path has no collective (requests shard across GPUs); what crosses
ranks is the timing: the job's time is the slowest rank's, and the reported
rate counts every rank's rows.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import numpy as np
    import torch.distributed as dist

    import bench
    from mla_latent_cache_absorbed_gb300 import workloads as W

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        # each rank's own batch: same shape, different values
        wl = W.make_workload("glm52_decode", seed=bench.rank_seed(rank))
        digest = float(np.asarray(wl.q_nope, np.float64).sum())
        # a deliberately uneven per-rank time: the job time is the maximum
        ms = 10.0 + 5.0 * rank
        ms_max = bench.max_over_ranks(ms, "cpu")
        rate = bench.whole_job_rate(wl.rows, w, 100, ms_max)
        out.put((rank, wl.rows, digest, ms_max, rate))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_and_sharding():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, rows0, d0, m0, v0), (r1, rows1, d1, m1, v1) = res
    assert rows0 == rows1                      # same batch shape on every rank
    assert d0 != d1                            # but independent inputs
    assert m0 == m1 == 15.0                    # the slowest rank's time
    assert v0 == v1 == pytest.approx(rows0 * 2 * 100 / 0.015)


def test_rank_zero_runs_the_named_workload():
    import bench
    assert bench.rank_seed(0) is None
    assert bench.rank_seed(1) != bench.rank_seed(2)
