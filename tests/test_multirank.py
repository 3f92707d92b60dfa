"""Host-side multi-rank logic of bench.py, on CPU with two gloo ranks.

The decode path shards by rows with no collective: every rank runs an independent
replica (own seed, own slots and inputs); the only cross-rank operations are the
barrier and the max of the timed interval. These tests run those operations with
world size 2 on 127.0.0.1."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import rssm_workloads as W
    d = bench.Dist()
    try:
        assert d.world == world and d.rank == rank and d.pg is not None
        d.barrier()
        # each rank reports its own elapsed time; everybody must see the max
        mine = 1.5 + rank
        got = d.max(mine)
        wl = W.mamba2_large(batch=8, nheads=4, ngroups=2, num_slots=16, steps=1,
                            seed=bench.shard_seed(0, rank))
        out[rank] = (got, wl.cache_indices().tolist(), float(wl.step_inputs(0)["x"].sum()))
    finally:
        d.close()


def test_two_rank_max_and_independent_replicas():
    ctx = mp.get_context("spawn")
    world = 2
    port = _free_port()
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 2.5
    # independent replicas: different slots and inputs per rank
    assert out[0][1] != out[1][1]
    assert out[0][2] != out[1][2]


def test_weak_scaling_value_sums_all_ranks():
    # value = ranks x rows per rank / max step time; a slower rank sets the time
    world, batch, ms_max = 4, 512, 0.2
    rows_s = world * batch / (ms_max * 1e-3)
    assert rows_s == pytest.approx(10.24e6)


def test_shard_seeds_are_distinct():
    import bench
    seeds = {bench.shard_seed(0, r) for r in range(8)}
    assert len(seeds) == 8
