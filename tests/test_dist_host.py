"""World-size-2 gloo test of the multi-GPU host logic (no GPU): each rank
serves a different batch, the step time is the max over ranks and the byte
total is the sum over ranks."""
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
    try:
        from paged_kv_cache_194_gb300 import replicas, workloads as wl
        w = replicas.rank_workload(wl.WORKLOADS["llama"], rank)
        lens = wl.seq_lens(w)
        t = replicas.max_over_ranks(1.0 + rank)          # rank 1 is the slower one
        total = replicas.sum_over_ranks(float(lens.sum()))
        out[rank] = (t, total, int(lens.sum()), w.seed)
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_reduce_on_gloo():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    (t0, tot0, n0, s0), (t1, tot1, n1, s1) = out[0], out[1]
    assert t0 == t1 == 2.0
    assert tot0 == tot1 == n0 + n1
    assert s0 != s1 and n0 != n1  # each rank serves its own batch
