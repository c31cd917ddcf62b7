"""Tensor-parallel shards on one GPU: two I-shards of the full-width block
(each with the replicated router and half of every expert's and of the shared
expert's intermediate columns) give fp32 partial outputs whose sum, formed by
moe_sum_partials through the C ABI, matches the full-width oracle."""
import numpy as np
import pytest
import torch

import moe_synth
from moe_decode_expert_gb300 import tp
from tests._util import check_tokens, oracle_sampled, oracle_tokens, parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def m():
    import __graft_entry__
    __graft_entry__.build()
    import moe_decode_expert_gb300 as mod
    return mod


@pytest.mark.parametrize("name,T", [("full_decode", 1), ("sharded_decode", 1), ("small_batch", 4)])
def test_two_shards_sum_to_the_full_block(m, name, T):
    wl = moe_synth.workload(name)
    cfg = m.cfg_from_workload(wl)
    G = 2
    scfg = tp.shard_cfg(cfg, G)
    g = moe_synth.make_layer(wl, 1, T, device=DEV)
    ws = m.alloc_workspace(scfg, T, DEV)
    partials = torch.full((G, T, wl.hidden), float("nan"), dtype=torch.float32, device=DEV)
    ids = torch.empty(G, T, wl.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(G, T, wl.top_k, dtype=torch.float32, device=DEV)
    for r in range(G):
        shard = tp.shard_layer(g, r, G, wl.inter, wl.shared_inter)
        tp.partial_forward(scfg, shard, g["x"], ids[r], w[r], partials[r], ws)
    out = torch.empty(T, wl.hidden, dtype=cfg.out_torch_dtype, device=DEV)
    m.moe_sum_partials(partials, out)
    res = torch.empty_like(out)
    m.moe_sum_partials(partials, res, residual=g["x"])
    m.moe_query_status(ws)
    assert torch.equal(ids[0], ids[1]) and torch.equal(w[0], w[1])  # every shard routes alike
    # the sum kernel: part order, one rounding; with the residual after the sum
    assert torch.equal(out, (partials[0] + partials[1]).to(out.dtype))
    assert torch.equal(res, ((partials[0] + partials[1]) + g["x"].float()).to(out.dtype))
    tokens = list(range(T))
    ref = oracle_tokens(wl, g, tokens)
    check_tokens(ids[0], w[0], partials[0] + partials[1], ref, tokens, wl.top_k)
    parity(out, ref["out"])


def test_sum_partials_rejects_bad_arguments(m):
    parts = torch.zeros(2, 12, device=DEV)
    with pytest.raises(m.MoeError) as ei:
        m.moe_sum_partials(parts, torch.empty(12, dtype=torch.bfloat16, device=DEV))  # n % 8 != 0
    assert ei.value.code == 1
