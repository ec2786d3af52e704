"""The multi-GPU benchmark runs independent replicas (no data-path collective); its only
cross-rank logic is the barrier and the max-over-ranks time.  Checked here with two CPU
ranks on the gloo backend."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    # rank r "took" 10 * (r + 1) ms for its steps; the job's time is the slowest rank's
    t = bench.max_over_ranks(ws, 10.0 * (rank + 1), device="cpu")
    v = bench.job_throughput(ws, 8, 5, t)
    out[rank] = (t, v)
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_max_time_and_job_throughput():
    ws = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:   # no fork of this (threaded) process
        out = m.dict()
        mp.start_processes(_worker, args=(ws, port, out), nprocs=ws, start_method="spawn")
        res = dict(out)
    assert res[0] == res[1]
    t, v = res[0]
    assert t == 20.0
    assert v == pytest.approx(2 * 8 * 5 / 0.020)
