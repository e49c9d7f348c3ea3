"""Multi-rank path of bench.py on the CPU: world-size-2 gloo ranks.

The hot path shards by request, so ranks share nothing on the data path;
the only cross-rank steps are the barrier and the max over ranks of the step
time, from which the whole-job throughput is computed.  Each rank also
serves its own requests (its own seed).
"""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import workload as wl
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    ms_local = 0.5 + rank            # rank 1 is the slower one
    bench.barrier(world)
    ms = bench.max_over_ranks(ms_local, world)
    rec = wl.CONFIGS["cfg2"].scaled(seed=wl.CONFIGS["cfg2"].seed + rank)
    q = rec.index_queries(1, 0, 1)
    results[rank] = (ms, int(q.astype("int64").sum()))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_distinct_requests():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert results[0][0] == results[1][0] == 1.5          # max over ranks
    assert results[0][1] != results[1][1]                 # each rank its own requests
    tokens_per_rank = 8 * 4
    value = 2 * tokens_per_rank / (results[0][0] * 1e-3)  # whole-job throughput
    assert value == pytest.approx(2 * 32 / 1.5e-3)
