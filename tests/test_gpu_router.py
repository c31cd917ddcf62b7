"""GPU parity of moe_router_topk (T >= 1) against the oracle and against an
exact ranking of the GPU's own fp32 logits."""
import numpy as np
import pytest
import torch

import moe_synth
import oracle
from tests._util import ocfg, min_rank_gap, fp32_topk

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def m():
    import __graft_entry__
    __graft_entry__.build()
    import moe_decode_expert_gb300 as mod
    return mod


def _route(m, cfg, x, wr):
    T = x.shape[0]
    ids = torch.full((T, cfg.top_k), -1, dtype=torch.int32, device=DEV)
    w = torch.full((T, cfg.top_k), float("nan"), dtype=torch.float32, device=DEV)
    lg = torch.full((T, cfg.n_experts), float("nan"), dtype=torch.float32, device=DEV)
    ws = m.alloc_workspace(cfg, T, DEV)
    m.moe_router_topk(cfg, x, wr, ids, w, ws, logits=lg)
    m.moe_query_status(ws)
    return ids.cpu().numpy(), w.cpu().numpy(), lg.cpu().numpy()


@pytest.mark.parametrize("name,T", [("tiny", 1), ("tiny", 37), ("full_decode", 1), ("full_decode", 64),
                                    ("chunked_prefill", 300), ("chunked_prefill", 1000), ("sharded_decode", 300)])
def test_router_matches_oracle(m, name, T):
    wl = moe_synth.workload(name)
    cfg = m.cfg_from_workload(wl)
    x = moe_synth.make_x(wl, 0, T, "cpu")
    wr = moe_synth.make_layer(wl, 0, 1, weights_only=True)["router_w"]
    ids, w, lg = _route(m, cfg, x.to(DEV), wr.to(DEV))
    c = ocfg(wl)
    xb, wrb = moe_synth.bits(x), moe_synth.bits(wr)
    # the selection itself is exact on the GPU's own fp32 logits
    assert np.array_equal(ids, fp32_topk(lg, wl.top_k))
    checked = 0
    for t in range(T):
        olg, oids, ow = oracle.router(c, xb[t], wrb)
        np.testing.assert_allclose(lg[t], olg, rtol=0, atol=1e-4 * max(1.0, np.abs(olg).max()))
        if min_rank_gap(olg, wl.top_k) > 1e-4:
            assert np.array_equal(ids[t], oids), t
            np.testing.assert_allclose(w[t], ow, rtol=1e-4, atol=1e-6)
            checked += 1
    assert checked >= max(1, int(0.9 * T))


@pytest.mark.parametrize("E,k", [(8, 3), (16, 2), (64, 8), (300, 20)])
def test_router_exact_ties(m, E, k):
    """Logits on a coarse dyadic grid are exact in fp32 too, so ties are real
    ties on both sides: ids must equal the oracle's (lower index first)."""
    H, T = 64, 40
    rng = np.random.default_rng(E * 31 + k)
    q = rng.integers(-2, 3, size=(E, H)) / 8.0
    wr = torch.from_numpy(q.astype(np.float32)).to(torch.float16)
    x = torch.ones(T, H, dtype=torch.float16)
    x[1::2] = 0.0                      # every other token: all logits 0
    cfg = m.MoeCfg(H, E, k, 8, 0, m.MOE_F16)
    ids, w, lg = _route(m, cfg, x.to(DEV), wr.to(DEV))
    c = oracle.OracleCfg(H, E, k, 8, 0, oracle.F16)
    for t in range(T):
        olg, oids, ow = oracle.router(c, moe_synth.bits(x)[t], moe_synth.bits(wr))
        assert np.array_equal(lg[t], olg.astype(np.float32))
        assert np.array_equal(ids[t], oids), (t, ids[t], oids)
        np.testing.assert_allclose(w[t], ow, rtol=2e-6)
    assert np.array_equal(ids[1], np.arange(k))


def test_router_without_renormalisation(m):
    wl = moe_synth.Workload("nr", 256, 16, 4, 8, 0, moe_synth.BF16, 0, 1.0, 0.05, 0.05, norm_topk=0,
                            preset_id=7)
    cfg = m.cfg_from_workload(wl)
    x = moe_synth.make_x(wl, 0, 20, "cpu")
    wr = moe_synth.make_layer(wl, 0, 1, weights_only=True)["router_w"]
    ids, w, lg = _route(m, cfg, x.to(DEV), wr.to(DEV))
    c = ocfg(wl)
    for t in range(20):
        olg, oids, ow = oracle.router(c, moe_synth.bits(x)[t], moe_synth.bits(wr))
        if min_rank_gap(olg, 4) > 1e-4:
            assert np.array_equal(ids[t], oids)
            np.testing.assert_allclose(w[t], ow, rtol=1e-5)
            assert w[t].sum() < 1.0
