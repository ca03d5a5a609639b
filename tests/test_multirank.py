"""The multi-rank benchmark path on CPU: two gloo ranks, max-over-ranks timing,
whole-job throughput and per-rank replicas (the path shards by sequence; each
rank owns its own batch and pool, no collective touches the data)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                  # rank 1 is the slowest
        got = bench.max_over_ranks(ms, world)
        gbps = bench.whole_job_gbps(1_000_000_000, world, 4, got)
        w = bench.replica_workload("tiny", rank)
        dist.barrier()
        results[rank] = (got, gbps, int(w.q[0, 0, 0, :4].astype(np.int64).sum()),
                         w.q.shape, w.num_blocks)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
        r = dict(results)
    assert r[0][0] == r[1][0] == 15.0                    # slowest rank's time on every rank
    assert r[0][1] == pytest.approx(2 * 4 * 1e9 / 15e-3 / 1e9)
    assert r[0][3] == r[1][3] and r[0][4] == r[1][4]     # replicas have the same shapes
    assert r[0][2] != r[1][2]                            # ... and their own data


def test_single_rank_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_gbps(2_000_000_000, 1, 10, 20.0) == pytest.approx(1000.0)
