"""The N > 1 host path of bench.py on CPU: two gloo ranks, as torchrun would start them.

The forward shards into independent replicas (every (batch, head) is
independent), so ranks share no data; only their timings meet, as a maximum
over ranks, and the whole-job value counts every rank's work.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import seeded_inputs as si


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's own timings; the slowest per entry must come back to every rank
        mine = [10.0 + rank, 5.0 - rank, 1.0 + 0.5 * rank]
        got = bench.max_over_ranks(mine, dist, "cpu")
        # each rank its own seeded batch: a digest of its K tensor
        q, k, v = si.make_qkv(1, 2, 2, 16, 64, seed=bench.replica_seed(rank))
        digest = int(np.bitwise_xor.reduce(k.reshape(-1).astype(np.uint64)))
        digests = [None] * world
        dist.all_gather_object(digests, digest)
        out[rank] = (got, digests)
    finally:
        dist.barrier()
        dist.destroy_process_group()


@pytest.mark.timeout(180)
def test_two_gloo_ranks_max_timing_and_independent_batches():
    world = 2
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert sorted(res) == [0, 1]
    for rank in range(world):
        got, digests = res[rank]
        assert got == [11.0, 5.0, 1.5]  # element-wise max over ranks
        assert digests[0] != digests[1]  # independent batches, no shared data


def test_whole_job_value_counts_every_rank():
    flops = 2.0 * 4 * 32 * 8192 ** 2 * 128
    one = bench.whole_job_tflops(1, flops, 2.0)
    assert bench.whole_job_tflops(2, flops, 2.0) == pytest.approx(2 * one)
    assert one == pytest.approx(flops / 2e-3 / 1e12)
    assert bench.max_over_ranks([3.0, 1.0], None, "cpu") == [3.0, 1.0]
