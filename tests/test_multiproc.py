"""The N > 1 path of bench.py on CPU: two gloo ranks (world size 2).

Each rank runs its own replica of the workload (sequences shard across GPUs with
no exchange), so the only cross-rank steps are the barrier and the reductions
of timings and byte counts. This checks them with torch.distributed on gloo:
the step time is the max over ranks, the work is the sum, and each rank's
replica is drawn from its own seed.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist
    import bench
    r, w = bench.dist_setup()
    assert (r, w) == (rank, world) and dist.get_backend() == "gloo"
    bench.barrier(w)
    ms = [3.0, 5.0][rank]                      # per-rank step time
    nbytes = [1.0e9, 2.0e9][rank]              # per-rank work
    ms_max = bench.reduce_over_ranks(ms, w, "max")
    total = bench.reduce_over_ranks(nbytes, w, "sum")
    # each rank's replica comes from its own seed: the paged histories differ
    import workloads as W
    c = W.make_paged(B=4, H=4, Hkv=2, dk=16, dv=16, block_size=4, num_blocks=40_000, seed=3 + 1000 * rank,
                     len_hi=64, mbps=17)
    lens = [int(x) for x in c.seq_lens]
    gathered = [None, None]
    dist.all_gather_object(gathered, lens)
    out.put((rank, ms_max, total, gathered))
    dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, total, gathered in res:
        assert ms_max == 5.0                  # the job takes as long as its slowest rank
        assert total == 3.0e9                 # value = work of all ranks / that time
        assert gathered[0] != gathered[1]     # distinct replicas per rank
