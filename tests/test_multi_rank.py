"""Host logic of the multi-GPU benchmark path on CPU with two gloo ranks: each rank takes a
different shard of the same varlen batch (disjoint query sets that together with the other
shards partition the batch), and the job time is the maximum over ranks."""
import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

import workloads as W
from oracle import split as osplit


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = W.WORKLOADS[bench.WORKLOAD_ID]
        shard = bench.shard_for_rank(rank, wl.sp)
        local = 1.0 + 0.25 * rank                       # pretend step time of this rank
        out[rank] = (shard, bench.max_over_ranks(local, dist, "cpu"))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_disjoint_shards_and_max_time():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    shards = [out[r][0] for r in range(world)]
    assert len(set(shards)) == world
    assert all(out[r][1] == 1.25 for r in range(world))
    wl = W.WORKLOADS[1]
    cu = W.cu_seqlens(wl.lengths)
    sets = [set(osplit.round_robin_split(cu, wl.sp, s)["gidx"].tolist()) for s in shards]
    assert not (sets[0] & sets[1])
    assert len(sets[0]) + len(sets[1]) == sum(len(osplit.round_robin_split(cu, wl.sp, s)["gidx"]) for s in shards)


def test_shard_assignment_covers_all_shards_for_eight_ranks():
    import bench
    wl = W.WORKLOADS[1]
    assert sorted(bench.shard_for_rank(r, wl.sp) for r in range(wl.sp)) == list(range(wl.sp))
    assert bench.shard_for_rank(0, wl.sp) == 3
