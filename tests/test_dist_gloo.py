"""Multi-process host logic of bench.py on CPU (gloo, world size 2): the step
time is the maximum over ranks and the value counts the work of every rank
(independent replicas; the path has no data exchange between GPUs)."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    dist.barrier()
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")   # rank 1 is the slow one
    out[rank] = (ms, bench.job_value(ws, 2.0e12, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_job_value_with_two_gloo_ranks():
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, _free_port(), out), nprocs=2, join=True)
    assert out[0] == out[1]
    ms, value = out[0]
    assert ms == pytest.approx(15.0)
    assert value == pytest.approx(2 * 2.0e12 / 15e-3 / 1e12)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.job_value(1, 1e12, 1000.0) == pytest.approx(1.0)
