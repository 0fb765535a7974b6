"""The N > 1 benchmark path on CPU: ranks run independent replicas over heads
and the job time is the maximum over ranks (gloo, world size 2, no GPU)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    ms = 10.0 + 5.0 * rank            # rank 1 is the slow one
    total = bench.reduce_max(ms, torch.device("cpu"))
    value = bench.job_value(step_flops=7e12, ms_per_step=total, world=w)
    out[rank] = (r, w, total, value)
    dist.destroy_process_group()


def test_two_rank_max_timing():
    world, port = 2, _free_port()
    mgr = tmp.Manager()
    out = mgr.dict()
    tmp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    res = dict(out)
    assert res[0][:2] == (0, 2) and res[1][:2] == (1, 2)
    # both ranks agree on the slowest rank's time; value counts both ranks' work
    assert res[0][2] == res[1][2] == 15.0
    assert res[0][3] == pytest.approx(2 * 7e12 / 15e-3 / 1e12)
