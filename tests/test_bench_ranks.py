"""The bench's multi-rank arithmetic on CPU: two gloo ranks on 127.0.0.1, each
timing its own replica of the step; both must report the maximum step time
over the ranks and the FLOPs of both ranks over that time.  No GPU."""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, ms, flops, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    dist.barrier()
    q.put((rank, *bench.aggregate_step(ms[rank], flops, world, "cpu")))
    dist.destroy_process_group()


def test_two_ranks_report_the_max_time_and_the_whole_job_value():
    world, flops = 2, 3.0e13
    ms = [100.0, 125.0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    mp.start_processes(_rank, args=(world, _free_port(), ms, flops, q), nprocs=world,
                       start_method="spawn", join=True)
    got = sorted(q.get(timeout=30) for _ in range(world))
    for rank, ms_max, value in got:
        assert ms_max == 125.0
        assert abs(value - world * flops / 0.125 / 1e12) < 1e-9


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.aggregate_step(50.0, 1.0e12, 1)
    assert ms == 50.0 and abs(value - 20.0) < 1e-12
