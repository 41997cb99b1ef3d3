"""The N > 1 path on CPU: two gloo ranks combine their step times the way
bench.py does for GPU replicas (max over ranks, whole-job token count)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from routed_expert_ffn_sigmoid_gb300 import replicas


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
        local_ms = [120.0, 150.0][rank]  # rank 1 is the slow replica
        value, ms_per_step = replicas.job_throughput(local_ms, tokens_per_rank_step=64, steps=10,
                                                     world=world)
        results[rank] = (value, ms_per_step, replicas.max_over_ranks(float(rank)))
    finally:
        dist.destroy_process_group()


def test_two_rank_job_throughput():
    world = 2
    manager = mp.Manager()
    results = manager.dict()
    mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
    for rank in range(world):
        value, ms_per_step, mx = results[rank]
        assert ms_per_step == pytest.approx(15.0)            # the slow rank's 150 ms / 10 steps
        assert value == pytest.approx(64 * 10 * 2 / 0.150)   # all tokens / job time
        assert mx == 1.0


def test_shard_range_partitions():
    for n in (0, 1, 7, 64, 4096):
        for world in (1, 2, 3, 8):
            spans = [replicas.shard_range(n, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1


def test_single_process_is_identity():
    assert replicas.max_over_ranks(3.5) == 3.5
    value, ms = replicas.job_throughput(100.0, 8, 4, 1)
    assert ms == 25.0 and value == pytest.approx(8 * 4 / 0.1)
