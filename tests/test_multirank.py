"""The bench's multi-rank logic on CPU with two gloo ranks: replicas get their
own seeds, the slowest rank's time is what every rank reports, and the
whole-job throughput counts every rank's batch."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
import workloads as W


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = bench.replica_workload(W.get("tiny"), rank)
        x = W.generate(w)
        step_ms = 1.0 + rank                       # the slower rank decides
        slowest = bench.reduce_max(step_ms, dist)
        value = bench.aggregate_tokens_per_s(world, w.batch, slowest)
        out[rank] = (w.seed, float(W.bf16_bits_to_f32(x.q).sum()), slowest, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    (s0, q0, t0, v0), (s1, q1, t1, v1) = res[0], res[1]
    assert s0 != s1 and q0 != q1                  # independent replicas
    assert t0 == t1 == 2.0                        # max over ranks
    assert v0 == v1 == pytest.approx(world * 1 / 2e-3)
