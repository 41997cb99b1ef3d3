"""Tensor parallelism along I on CPU: two gloo ranks each compute the layer on
their slice of every expert's intermediate dimension (the oracle on the
slices of tests/tp_slices.py), then exchange the fp32 partial outputs with
the library's own exchange step (tensor_parallel.sum_partials): all-reduce,
and reduce-scatter of token rows.  The sum must equal the unsplit layer.

The split is the compute form of the pages' dual-GPU placement ("GLM5next
Production Readiness: Optional Mix Qtypes + Cache Allocation", UNIT 2:
Dual-GPU Placement)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import oracle
import synthetic
from moe_inputs import make_inputs
from tp_slices import slice_stack

WORKLOADS = {"bf16": synthetic.WORKLOADS["tiny"],
             "int4": synthetic.Workload("tiny_int4", 8, 256, 288, 256, 256, 8, "int4", 5,
                                        tokens=(8,))}


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, fmt, results):
    import torch
    import torch.distributed as dist

    from routed_expert_ffn_sigmoid_gb300 import tensor_parallel as tp

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = make_inputs(WORKLOADS[fmt])
        ex = slice_stack(inp.experts, rank, world)
        sh = slice_stack(inp.shared, rank, world)
        part, idx, _ = oracle.moe_forward(inp.x, inp.w_router, inp.b_router, ex, sh, fmt)
        full = torch.from_numpy(part.astype(np.float32))
        rows = tp.sum_partials(full.clone(), scatter_rows=True)
        summed = tp.sum_partials(full)
        results[rank] = (summed.numpy(), rows.numpy(), idx)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("fmt", ["bf16", "int4"])
def test_two_rank_split_along_I_sums_to_the_layer(fmt):
    world = 2
    manager = mp.Manager()
    results = manager.dict()
    mp.spawn(_worker, args=(world, _free_port(), fmt, results), nprocs=world, join=True)
    inp = make_inputs(WORKLOADS[fmt])
    ref, ref_idx, _ = oracle.moe_forward(inp.x, inp.w_router, inp.b_router, inp.experts,
                                         inp.shared, fmt)
    rms = float(np.sqrt(np.mean(ref * ref)))
    T = ref.shape[0]
    for rank in range(world):
        summed, rows, idx = results[rank]
        assert np.array_equal(idx, ref_idx)  # every part routes identically
        # fp32 partials: the sum is the layer within fp32 rounding
        assert np.max(np.abs(summed - ref)) / rms <= 1e-6
        a, b = rank * T // world, (rank + 1) * T // world
        assert np.array_equal(rows, summed[a:b])


def test_slices_partition_the_stack():
    # the parts' slices tile every matrix exactly
    for fmt, wl in WORKLOADS.items():
        st = synthetic.gen_experts(wl, e0=0, e1=3)
        for parts in (1, 2, 4):
            sl = [slice_stack(st, p, parts) for p in range(parts)]
            for name in st:
                axis = 2 if name.startswith("down") else 1
                assert np.array_equal(np.concatenate([s[name] for s in sl], axis=axis), st[name])
