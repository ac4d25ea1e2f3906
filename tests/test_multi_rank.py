"""Host logic of the multi-GPU benchmark path on CPU with two gloo ranks: every rank runs an
independent replica of the whole many-request batch (all of its shards, which partition the
batch's tokens), so the job processes world x the batch's queries, and the job time is the
maximum over ranks."""
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
        shards = bench.shards_for_rank(rank, world, wl.sp)
        local = 1.0 + 0.25 * rank                       # pretend step time of this rank
        out[rank] = (tuple(shards), bench.max_over_ranks(local, dist, "cpu"))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_run_whole_replicas_and_max_time():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    assert all(out[r][1] == 1.25 for r in range(world))
    import bench
    wl = W.WORKLOADS[bench.WORKLOAD_ID]
    cu = W.cu_seqlens(wl.lengths)
    for r in range(world):
        shards = out[r][0]
        assert sorted(shards) == list(range(wl.sp))
        # the shards of one replica partition the batch's tokens
        sets = [set(osplit.round_robin_split(cu, wl.sp, s)["gidx"].tolist()) for s in shards]
        assert sum(len(x) for x in sets) == int(cu[-1])
        assert set().union(*sets) == set(range(int(cu[-1])))


def test_default_workload_is_the_many_request_batch():
    import bench
    wl = W.WORKLOADS[bench.WORKLOAD_ID]
    assert len(wl.lengths) == 32 and sum(wl.lengths) == 71014 and wl.sp == 4
    assert list(wl.ranks) == [0, 1, 2, 3]
