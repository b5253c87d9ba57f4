"""The benchmark's multi-rank logic on CPU: two gloo ranks on 127.0.0.1.
Each rank runs its own independent problem (the attention forward shards
over heads and batches with no exchange), so the only cross-rank operations
are a barrier and the max over ranks of the timed region."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench._barrier(world)
    t = bench._max_over_ranks(10.0 + rank, world, torch.device("cpu"))
    out[rank] = t
    bench._barrier(world)
    dist.destroy_process_group()


def test_two_gloo_ranks_max_and_barrier():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 11.0


def test_whole_job_aggregate():
    import bench
    # 2 ranks x 5 steps x 1e12 FLOP in 10 ms (slowest rank) -> 1000 TFLOPS
    assert bench.whole_job_tflops(1e12, 2, 10.0, 5) == pytest.approx(1000.0)
    assert bench.whole_job_tflops(1e12, 1, 10.0, 5) == pytest.approx(500.0)
