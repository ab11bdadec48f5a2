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


# ------------------------------------------------------------- head partition
def _shard_rank(rank, world, port, q):
    """One rank of a head-sharded layer: its own heads through the fp64
    oracle, gathered on every rank; the timing reduction of the bench."""
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import numpy as np

    import bench
    from block_sparse_gated_gb300 import workloads as wl
    from block_sparse_gated_gb300.shard import head_shard, shard_tensors
    from oracle import bsfa_oracle as orc
    Hq, Hkv, L, d, B = 8, 4, 300, 16, 64
    x = wl.layer_inputs(Hq, Hkv, L, d, 77, skip_rate=0.3)  # every rank draws the same layer
    T = torch.full((2, Hq, 3), 0.4)
    T[1] = torch.linspace(0.1, 0.9, Hq * 3).reshape(Hq, 3)
    sh = head_shard(Hq, Hkv, rank, world)
    qs, ks, vs, ts = shard_tensors(sh, x.q, x.k, x.v, T)
    r = orc.prefill(qs.double().numpy(), ks.double().numpy(), vs.double().numpy(), Bq=B, Bk=B,
                    thresholds=ts[1].double().numpy())
    parts = [None] * world
    dist.all_gather_object(parts, (list(sh.q_heads), ts[1].tolist(), r["out"], r["keep"]))
    ms, value, total = bench.aggregate_shards([80.0, 100.0][rank], [1.0e13, 3.0e13][rank], world,
                                              "cpu")
    if rank == 0:
        full = orc.prefill(x.q.double().numpy(), x.k.double().numpy(), x.v.double().numpy(),
                           Bq=B, Bk=B, thresholds=T[1].double().numpy())
        heads = [h for p in parts for h in p[0]]
        rows = [row for p in parts for row in p[1]]
        out = np.concatenate([p[2] for p in parts])
        keep = np.concatenate([p[3] for p in parts])
        q.put((heads, rows, T[1].tolist(), float(np.abs(out - full["out"]).max()),
               bool(np.array_equal(keep, full["keep"])), ms, value, total))
    dist.destroy_process_group()


def test_head_shards_cover_the_layer_once_and_reduce_the_timing():
    """Two gloo ranks split 4 KV heads (8 query heads): every query head is
    computed exactly once, each rank's threshold rows are its own heads'
    rows, the concatenated shards equal the unsharded layer (fp64 oracle),
    and the step time is the max over ranks with the FLOPs summed."""
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    mp.start_processes(_shard_rank, args=(world, _free_port(), q), nprocs=world,
                       start_method="spawn", join=True)
    heads, rows, T_full, err, same_keep, ms, value, total = q.get(timeout=60)
    assert heads == list(range(8))
    assert rows == T_full
    assert err == 0.0 and same_keep
    assert ms == 100.0 and total == 4.0e13
    assert abs(value - 4.0e13 / 0.1 / 1e12) < 1e-9


def test_head_shard_split_rules():
    sys.path.insert(0, ROOT)
    import pytest

    from block_sparse_gated_gb300.shard import head_shard
    # Llama-3.1-8B: 32 query heads over 8 KV heads, for 1, 2, 4 and 8 ranks
    for world in (1, 2, 4, 8):
        got = [head_shard(32, 8, r, world) for r in range(world)]
        assert [h for s in got for h in s.q_heads] == list(range(32))
        assert [h for s in got for h in s.kv_heads] == list(range(8))
        assert all(len(s.kv_heads) == 8 // world for s in got)
        for s in got:  # each query head reads a KV head of its own rank
            assert all(h // 4 in s.kv_heads for h in s.q_heads)
    # uneven: 5 KV heads over 3 ranks -> 2, 2, 1
    assert [len(head_shard(10, 5, r, 3).kv_heads) for r in range(3)] == [2, 2, 1]
    with pytest.raises(ValueError):
        head_shard(32, 8, 0, 16)  # a KV head is never split
    with pytest.raises(ValueError):
        head_shard(32, 8, 2, 2)
