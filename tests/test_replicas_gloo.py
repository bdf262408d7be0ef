"""The multi-GPU form of the benchmark is N independent replicas (the decode
path has no exchange step): each rank draws its own batch, and the job's
figures are the slowest rank's time and the sum of all ranks' tokens.  This
checks that host logic with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from paged_kv_cache_179_gb300 import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = W.make_workload("tiny", seed=bench.replica_seed(7, rank),
                            lens_override=[5 + rank, 40, 77, 300])
        step_ms = 10.0 + 5.0 * rank            # rank 1 is the slower one
        e2e_ms = 20.0 - 3.0 * rank
        got = bench.reduce_over_ranks(step_ms, e2e_ms, w.total_tokens(), world, torch.device("cpu"))
        q.put((rank, got, w.total_tokens(), float(w.q.float().sum())))
    finally:
        dist.destroy_process_group()


def test_two_replicas_reduce_max_time_and_sum_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, got0, tok0, qs0), (r1, got1, tok1, qs1) = res
    assert got0 == got1                         # every rank sees the job's figures
    assert got0 == (15.0, 20.0, float(tok0 + tok1))
    assert qs0 != qs1                           # the replicas drew different batches


def test_single_rank_is_identity():
    assert bench.reduce_over_ranks(3.0, 4.0, 17, 1, torch.device("cpu")) == (3.0, 4.0, 17.0)
