"""Tensor parallelism of the MoE FFN layer along the expert intermediate size.

The pages' dual-GPU plan places experts on two GPUs ("GLM5next Production
Readiness: Optional Mix Qtypes + Cache Allocation", lucebox PR #2, section
"UNIT 2: Dual-GPU Placement").  The compute form of a split that keeps every
GPU equally loaded, whatever the routing skew, cuts the intermediate
dimension I of every expert (routed and shared) into ``parts`` slices:

* the clamped SwiGLU is elementwise in I, so part p needs rows
  [p Is, (p+1) Is) of gate and up and the same columns of down (Is = I/parts);
* every part routes identically (the router is replicated), runs
  ``moe_ffn_forward`` with I = I_shared = Is on its slices, and produces a
  partial fp32 output;
* the layer's output is the sum of the parts: one all-reduce, or one
  reduce-scatter when each rank continues with its own rows.

``slice_stack`` copies a part's weights through the library
(``moe_tp_slice_weights``, copy engine); ``sum_partials`` is the exchange
step, on any torch.distributed process group (NCCL across GPUs, gloo on CPU).
"""
from __future__ import annotations

import routed_expert_ffn_sigmoid_gb300 as moe


def slice_shapes(fmt: str, n_experts: int, H: int, I: int, parts: int) -> dict:
    """Shapes (and numpy-style dtypes) of one part's buffers: name -> (shape, dtype)."""
    Is = I // parts
    if fmt == "bf16":
        return {"gate": ((n_experts, Is, H), "int16"), "up": ((n_experts, Is, H), "int16"),
                "down": ((n_experts, H, Is), "int16")}
    return {"gate": ((n_experts, Is, H // 2), "uint8"), "up": ((n_experts, Is, H // 2), "uint8"),
            "down": ((n_experts, H, Is // 2), "uint8"),
            "gate_scale": ((n_experts, Is, H // 32), "int16"),
            "up_scale": ((n_experts, Is, H // 32), "int16"),
            "down_scale": ((n_experts, H, Is // 32), "int16")}


def slice_stack(dims, n_experts: int, part: int, parts: int, full: dict, stream=None):
    """Part ``part`` of ``parts`` of a weight stack, as new device tensors.

    ``dims`` are the full layer's dims; ``full`` maps gate/up/down (and the
    Int4 *_scale names) to the stack's device tensors.  Returns
    (tensors, moe_weights) for the slice.
    """
    import torch

    fmt = "bf16" if dims.fmt == moe.MOE_W_BF16 else "int4"
    dev = full["gate"].device
    tdt = {"int16": torch.int16, "uint8": torch.uint8}
    out = {name: torch.empty(shape, dtype=tdt[dt], device=dev)
           for name, (shape, dt) in slice_shapes(fmt, n_experts, dims.H, dims.I, parts).items()}
    src = moe.make_weights(full["gate"], full["up"], full["down"], full.get("gate_scale"),
                           full.get("up_scale"), full.get("down_scale"))
    dst = moe.make_weights(out["gate"], out["up"], out["down"], out.get("gate_scale"),
                           out.get("up_scale"), out.get("down_scale"))
    moe.moe_tp_slice_weights(dims, n_experts, part, parts, src, dst, stream)
    return out, dst


def part_dims(dims, parts: int):
    """The dims one part runs the layer with: I = I_shared = I / parts."""
    Is = dims.I // parts
    return moe.MoeDims(dims.T, dims.H, dims.E, Is, Is, dims.top_k, dims.fmt, dims.flags)


def sum_partials(out, group=None, scatter_rows: bool = False):
    """The exchange step: the sum over ranks of each rank's partial output.

    out [T][H] fp32 is this rank's partial.  With scatter_rows=False it is
    all-reduced in place and returned; with scatter_rows=True each rank gets
    the summed rows of its own share of the T tokens (contiguous, in rank
    order, the first T % world ranks one row more), through one
    reduce-scatter where the backend has it, else an all-reduce and a slice.
    """
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    if world == 1:
        return out
    if not scatter_rows:
        dist.all_reduce(out, op=dist.ReduceOp.SUM, group=group)
        return out
    from routed_expert_ffn_sigmoid_gb300.replicas import shard_range

    rank = dist.get_rank(group)
    T = out.shape[0]
    spans = [shard_range(T, r, world) for r in range(world)]
    if all(b - a == spans[0][1] - spans[0][0] for a, b in spans) and \
            dist.get_backend(group) == "nccl":
        mine = torch.empty((spans[rank][1] - spans[rank][0],) + tuple(out.shape[1:]),
                           dtype=out.dtype, device=out.device)
        dist.reduce_scatter_tensor(mine, out.contiguous(), op=dist.ReduceOp.SUM, group=group)
        return mine
    dist.all_reduce(out, op=dist.ReduceOp.SUM, group=group)
    a, b = spans[rank]
    return out[a:b].clone()
