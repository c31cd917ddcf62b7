"""Tensor-parallel use of the MoE block: weight sharding along the expert
intermediate dimension, the per-layer sum of partial outputs, and the
all-reduce that carries it across GPUs.

The pages run their model with TP = 4 ("BI-V100 inference work log", Part 2:
each expert's I = 512 split into 128 per GPU) and pay one all-reduce of the
MoE output per layer (Part 9; "Decode throughput analysis report", module
profiling).  Shard r of G holds, for every expert, gate rows and up rows
[r*I/G, (r+1)*I/G) of W13 and the same columns of W2, the same slices of the
shared expert, and the full router and shared-gate vector.  Every shard routes
the token itself (identical ids and weights) and emits an fp32 partial output;
the partials sum to the block's output.

Host-side pieces only: slicing (torch ops on the caller's device), the
all-reduce (torch.distributed, NCCL on GPUs), and the final sum/rounding
through the library's ``moe_sum_partials`` kernel.
"""
from __future__ import annotations

from dataclasses import replace

import torch

from . import MOE_F32, MoeCfg, moe_decode_forward, moe_grouped_forward, moe_sum_partials


def shard_cfg(cfg: MoeCfg, world: int) -> MoeCfg:
    """Config of one of ``world`` shards: I/world, Is/world, fp32 partial out."""
    if cfg.inter % world or cfg.shared_inter % world:
        raise ValueError("inter and shared_inter must divide by the shard count")
    c = replace(cfg, inter=cfg.inter // world, shared_inter=cfg.shared_inter // world, out_dtype=MOE_F32)
    if c.inter % 8 or c.shared_inter % 8:
        raise ValueError("each shard's inter and shared_inter must be multiples of 8")
    return c


def shard_layer(layer: dict, rank: int, world: int, inter: int, shared_inter: int) -> dict:
    """Shard ``rank`` of ``world`` of one layer's weights (contiguous copies).
    ``layer`` holds router_w [E, H], w13 [E, 2I, H], w2 [E, H, I], shared_w13
    [2Is, H] or None, shared_w2 [H, Is] or None, shared_gate_w [H] or None."""
    i0, i1 = rank * inter // world, (rank + 1) * inter // world
    w13 = layer["w13"]
    out = {
        "router_w": layer["router_w"],
        "w13": torch.cat([w13[:, i0:i1], w13[:, inter + i0:inter + i1]], dim=1).contiguous(),
        "w2": layer["w2"][:, :, i0:i1].contiguous(),
        "shared_gate_w": layer.get("shared_gate_w"),
        "shared_w13": None,
        "shared_w2": None,
    }
    if shared_inter:
        s0, s1 = rank * shared_inter // world, (rank + 1) * shared_inter // world
        sw13 = layer["shared_w13"]
        out["shared_w13"] = torch.cat([sw13[s0:s1], sw13[shared_inter + s0:shared_inter + s1]]).contiguous()
        out["shared_w2"] = layer["shared_w2"][:, s0:s1].contiguous()
    return out


def partial_forward(scfg: MoeCfg, shard: dict, x, ids, weights, partial, ws, stream=None):
    """This shard's fp32 partial output for x [T, H] (T = 1: the single-launch
    decode kernel; T > 1: the grouped path)."""
    f = moe_decode_forward if x.shape[0] == 1 else moe_grouped_forward
    f(scfg, x, shard["router_w"], shard["w13"], shard["w2"], shard["shared_w13"], shard["shared_w2"],
      shard["shared_gate_w"], ids, weights, partial, ws, stream)


def all_reduce_partials(partial: torch.Tensor, group=None):
    """Sum the shards' fp32 partial outputs in place across the process group
    (NCCL on GPUs, gloo on the CPU)."""
    import torch.distributed as dist
    dist.all_reduce(partial, op=dist.ReduceOp.SUM, group=group)
    return partial


def finish(partial_sum: torch.Tensor, out: torch.Tensor, residual=None, stream=None):
    """Round the summed fp32 output once into ``out`` (adding the residual
    first when given), through the library's kernel."""
    moe_sum_partials(partial_sum.reshape(1, *out.shape), out, residual, stream)
