"""World-size-2 gloo test of the benchmark's multi-rank host logic (CPU only).

Every rank runs its own copy of the workload (weak scaling, no data-path
collective); the step time is the maximum over ranks and the reported value is
the units all ranks processed over that time.
"""
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


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    local_ms = 10.0 + 5.0 * rank          # rank 1 is slower
    t = bench.max_over_ranks(local_ms, world)
    value = bench.aggregate_value(1_000_000_000, t, world)
    # per-rank workloads differ only by seed: same shapes and byte counts
    w = bench.rank_workload(rank)
    nbytes = sum(bench.compress_bytes(w.for_layer(l), w.batch * w.seq_len) for l in range(w.layers))
    out[rank] = (t, value, nbytes)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time_and_sum_work():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] == res[1][1] == pytest.approx(2 * 1e9 / 15e-3 / 1e9)
    assert res[0][2] == res[1][2] > 0
