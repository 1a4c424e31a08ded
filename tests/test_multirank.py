"""The multi-GPU benchmark path on CPU: two gloo ranks, each with its own
replica of the work; the job value is the sum of the ranks' FLOPs over the
slowest rank's time (max-reduced), with no other cross-rank traffic."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r did 1e12 FLOPs in (r + 1) * 100 ms
    tflops, ms = bench.job_throughput(1e12, (rank + 1) * 100.0, dist)
    out[rank] = torch.tensor([tflops, ms])
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        tflops, ms = out[r].tolist()
        assert ms == pytest.approx(200.0)          # slowest rank
        assert tflops == pytest.approx(2e12 / 0.2 / 1e12)


def test_single_process_aggregation():
    import bench
    tflops, ms = bench.job_throughput(5e11, 250.0)
    assert ms == 250.0 and tflops == pytest.approx(2.0)
