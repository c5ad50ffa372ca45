"""Host-side logic of the sharded (N > 1) bench path, with two gloo ranks on CPU.

Each rank owns an independent shard of the workload (no data exchange); the only collective
is the all-reduce that takes the slowest rank's step time.
"""

import os
import socket

import numpy as np
import pytest

import bench
from exact_tiled_attention_07_gb300.inputs import WORKLOADS, make_inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step_ms = [3.0, 5.0][rank]
        got = bench.max_over_ranks(step_ms, dist, "cpu")
        w = WORKLOADS["tiny_fp32"]
        shard = make_inputs(bench.shard_workload(w, rank))
        results[rank] = (got, float(shard["q"].sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step_and_own_distinct_shards():
    import torch.multiprocessing as mp

    manager = mp.get_context("spawn").Manager()
    results = manager.dict()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, results), nprocs=2, join=True, start_method="spawn")
    assert results[0][0] == 5.0 and results[1][0] == 5.0
    assert results[0][1] != results[1][1]


def test_aggregate_and_single_process():
    assert bench.max_over_ranks(4.5) == 4.5
    # two ranks, 1e12 FLOP each in 2 ms per step -> 1000 TFLOP/s for the job
    assert bench.aggregate_tflops(1e12, 2, 2.0) == pytest.approx(1000.0)
    w = WORKLOADS["tiny_fp32"]
    a = make_inputs(bench.shard_workload(w, 0))["q"]
    b = make_inputs(bench.shard_workload(w, 0))["q"]
    np.testing.assert_array_equal(a, b)
    assert bench.shard_workload(w, 0).seed == w.seed
