"""The N > 1 path of bench.py on CPU: two ranks over gloo on 127.0.0.1.

The fixed-size cache shards by sequence with no exchange step, so `bench.py --gpus N`
runs N independent replicas (weak scaling).  What N ranks share is bookkeeping: every
rank draws its own inputs, the timing is the slowest rank's, and the whole-job value
counts every rank's tokens.  These tests run that bookkeeping in two real processes
with the gloo backend (no GPU).
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from fixed_size_kv_gb300 import inputs
        cpu = torch.device("cpu")
        # each rank's own (made-up) step time: the job is as slow as the slowest rank
        local_ms = 100.0 + 25.0 * rank
        worst = bench.max_over_ranks(local_ms, world, cpu)
        value = bench.job_throughput(1000, world, worst)
        # independent replicas: each rank draws its own prompt lengths and inputs
        mixed = inputs.WORKLOADS["gqa_mixed_b64"]
        lengths = inputs.prompt_lengths(mixed, bench.replica_seed(0, rank), n=8)
        tiny = inputs.WORKLOADS["gqa_2k_tiny"]
        pre = inputs.gen_prefill(tiny, 64, seed=bench.replica_seed(0, rank), seq=0)
        k_sum = float(pre.K.float().sum())
        dist.barrier()
        results[rank] = (worst, value, tuple(lengths), k_sum)
    finally:
        dist.destroy_process_group()


@pytest.fixture(scope="module")
def two_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True,
                       start_method="spawn")
    return dict(results)


def test_timing_is_the_slowest_rank(two_ranks):
    assert two_ranks[0][0] == two_ranks[1][0] == 125.0


def test_whole_job_value_counts_every_rank(two_ranks):
    # 1000 tokens on each of 2 ranks over the slowest rank's 125 ms
    assert two_ranks[0][1] == two_ranks[1][1] == pytest.approx(2 * 1000 / 0.125)


def test_replicas_draw_independent_inputs(two_ranks):
    assert two_ranks[0][2] != two_ranks[1][2]
    assert two_ranks[0][3] != two_ranks[1][3]
