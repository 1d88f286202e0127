"""The multi-GPU bench path on CPU: two gloo ranks.

Decode attention shards by sequence with no exchange, so a multi-GPU run gives
every rank its own batch and reduces only the timings.  These checks run the
host side of that: each rank's shard differs from the others', the timing taken
is the slowest rank's, and the whole-job figure counts every rank's bytes.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from decode_attention_02_gb300 import inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.0, 5.0][rank]
        got = bench.max_over_ranks(ms, dist, torch.device("cpu"))
        w = bench.rank_workload(inputs.WORKLOADS["tiny_b1_l512_bf16"], rank)
        case = inputs.generate(w)
        dist.barrier()
        results[rank] = (got, w.seed, float(case.q.float().sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_and_shard_the_data():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:
        results = m.dict()
        mp.start_processes(_rank_main, args=(world, port, results), nprocs=world, start_method="spawn")
        r = dict(results)
    assert r[0][0] == r[1][0] == 5.0
    assert r[0][1] != r[1][1]                  # each rank decodes its own sequences
    assert r[0][2] != r[1][2]
    assert bench.whole_job_gbs(10 ** 9, world, 5.0) == pytest.approx(2 * 10 ** 9 / 5e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(4.0, None, None) == 4.0
    w = inputs.WORKLOADS["b32_l4096_bf16"]
    assert bench.rank_workload(w, 0) is w
