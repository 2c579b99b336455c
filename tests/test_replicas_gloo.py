"""The multi-rank (replicas) path of the benchmark on CPU: two gloo ranks, each
with its own synthetic batch, max-over-ranks timing and the whole-job rate."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    from token_dispatch_gb300 import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env()[:2] == (rank, world)
        # each rank its own batch (seed = rank), the same weights
        x, _ = synth.router_inputs(synth.TINY_F32, seed=rank)
        ms, e2e = bench.max_over_ranks([1.0 + rank, 5.0 - rank], "cpu")
        out[rank] = (float(x.ref[0, 0]), ms, e2e,
                     bench.whole_job_tokens_per_s(synth.TINY_F32.T, world, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_tokens():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    x0, ms0, e0, v0 = res[0]
    x1, ms1, e1, v1 = res[1]
    assert x0 != x1  # different batches per rank
    assert ms0 == ms1 == 2.0 and e0 == e1 == 5.0  # max over ranks
    assert v0 == v1 == pytest.approx(2 * 256 / 2e-3)  # both ranks' tokens over the slowest step
