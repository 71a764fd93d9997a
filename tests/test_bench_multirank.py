"""The multi-rank bench logic (replicas only: barrier, max over ranks,
whole-job rate) on world_size 2 with the gloo backend, on CPU."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, _ = bench._dist()
    assert (ws, r) == (world, rank)
    my_ms = 100.0 + 50.0 * rank            # rank 1 is slower
    dist.barrier()
    ms = bench.reduce_max(my_ms, dist, "cpu")
    out[rank] = (ms, bench.whole_job_rate(10_000, ws, ms))
    dist.destroy_process_group()


def test_two_rank_max_and_rate():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0][0] == out[1][0] == 150.0
    # 2 ranks x 10,000 tokens over the slowest rank's 150 ms
    assert out[0][1] == pytest.approx(2 * 10_000 / 0.150)


def test_single_rank_identity():
    import bench
    assert bench.reduce_max(12.5, None, "cpu") == 12.5
    assert bench.whole_job_rate(10_000, 1, 1000.0) == 10_000
