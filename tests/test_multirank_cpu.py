"""The multi-rank logic of bench.py on CPU: two gloo ranks on 127.0.0.1."""
import os
import socket

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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from workloads import WORKLOADS
    w = WORKLOADS["tiny"]
    ws, r, local = bench.dist_env()
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, torch.device("cpu"))
    seed = bench.rank_workload(w, rank).seed
    dist.barrier()
    out[rank] = (ws, r, local, ms, seed)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0][:3] == (2, 0, 0) and out[1][:3] == (2, 1, 1)
    assert out[0][3] == out[1][3] == 15.0           # max over ranks
    assert out[0][4] != out[1][4]                   # each rank its own batch


def test_job_throughput_counts_every_rank():
    import bench
    assert bench.job_tokens_per_s(1000, 4, 10, 2000.0) == pytest.approx(20000.0)
    assert bench.job_tokens_per_s(1000, 1, 10, 2000.0) == pytest.approx(5000.0)
