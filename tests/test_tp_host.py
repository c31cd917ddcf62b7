"""Host plumbing of tensor-parallel use on the CPU: sharding the weights along
the intermediate dimension and summing the shards' partial outputs with an
all-reduce over two gloo ranks gives the full-width block (the partials come
from the oracle, run on each rank's shard)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import moe_synth
import oracle
from moe_decode_expert_gb300 import tp


def _wl():
    return moe_synth.Workload("tp", 64, 8, 2, 32, 16, moe_synth.BF16, 1, 1.0, 0.1, 0.2, preset_id=7)


def _oracle(wl, d, I, Is):
    b = moe_synth.bits
    c = oracle.OracleCfg(wl.hidden, wl.n_experts, wl.top_k, I, Is, wl.dtype, wl.norm_topk, wl.has_shared_gate)
    return oracle.moe_forward(c, b(d["x"]), b(d["router_w"]), b(d["w13"]), b(d["w2"]), b(d["shared_w13"]),
                              b(d["shared_w2"]), b(d["shared_gate_w"]))


def test_shard_slices_are_the_intermediate_columns():
    wl = _wl()
    d = moe_synth.make_layer(wl, 0, 1)
    s1 = tp.shard_layer(d, 1, 2, wl.inter, wl.shared_inter)
    assert torch.equal(s1["w13"][:, :16], d["w13"][:, 16:32])           # gate rows 16..31
    assert torch.equal(s1["w13"][:, 16:], d["w13"][:, 48:64])           # up rows 48..63
    assert torch.equal(s1["w2"], d["w2"][:, :, 16:32])
    assert torch.equal(s1["shared_w13"], torch.cat([d["shared_w13"][8:16], d["shared_w13"][24:32]]))
    assert torch.equal(s1["shared_w2"], d["shared_w2"][:, 8:16])
    assert s1["router_w"] is d["router_w"] and s1["shared_gate_w"] is d["shared_gate_w"]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = _wl()
        T = 3
        d = moe_synth.make_layer(wl, 0, T)
        shard = tp.shard_layer(d, rank, world, wl.inter, wl.shared_inter)
        part = _oracle(wl, {**shard, "x": d["x"]}, wl.inter // world, wl.shared_inter // world)
        partial = torch.from_numpy(part["out"]).contiguous()
        tp.all_reduce_partials(partial)
        full = _oracle(wl, d, wl.inter, wl.shared_inter)
        q.put((rank, part["ids"].tolist(), full["ids"].tolist(),
               float(np.abs(partial.numpy() - full["out"]).max()), float(np.abs(full["out"]).max())))
    finally:
        dist.destroy_process_group()


def test_two_rank_all_reduce_of_shard_partials_gives_the_full_block():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ids, full_ids, err, mx in res:
        assert ids == full_ids            # every shard routes like the full block
        assert err <= 1e-12 * mx          # fp64 partials sum to the full output

