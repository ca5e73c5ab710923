"""Multi-rank bench logic on CPU: two gloo ranks, one replica each (the path
shards by independent batches, so the only exchange is the timing reduction)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    env = bench.dist_env()
    local_ms = 10.0 + 7.5 * rank           # rank 1 is the slow one
    q.put((rank, env, bench.max_over_ranks(local_ms, ws), bench.replica_seed(3, rank)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_reduction_and_replicas():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, mx, seed in res:
        assert env == (ws, rank, rank)
        assert mx == 17.5                   # every rank sees the max over ranks
    assert res[0][3] != res[1][3]           # distinct replicas


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25
