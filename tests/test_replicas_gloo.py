"""The multi-rank bench harness on CPU: two gloo ranks, rendezvous on 127.0.0.1.

The decode path shards by request with no exchange between GPUs, so N GPUs run N
independent replicas; the only cross-rank step is taking the slowest rank's
time.  This checks that step with real process groups, without a GPU.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = 10.0 + 5.0 * rank           # rank 1 is the slow replica
    got = bench.max_over_ranks(mine, "cpu")
    dist.barrier()
    out[rank] = got
    dist.destroy_process_group()


def test_slowest_rank_time_is_reported_by_every_rank():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5


def test_algorithmic_accounting_of_the_tiny_workload():
    import bench
    from workloads import mla as W
    p = W.config_tiny()
    alg = bench.algorithmic(p)
    keys = 37 + 70                                  # causal, one query at the end of each cache
    assert alg["keys"] == keys
    assert alg["kv_bytes"] == keys * 2 * (64 + 16)
    pages = 3 + 5
    assert alg["decode_bytes"] == alg["kv_bytes"] + 4 * pages
    w = 2 * (4 * 64 * 32 + 4 * 32 * 64)
    assert alg["total_bytes"] == alg["decode_bytes"] + w + 2 * 4 * 48 * 2 + 2 * 4 * 32 * 2
    flops = 2 * 4 * keys * 80 + 2 * 4 * keys * 64 + 2 * 2 * 4 * 64 * 32 + 2 * 2 * 4 * 32 * 64
    assert alg["flops"] == flops
