"""GPU parity of moe_grouped_forward (T > 1: device-side grouping per expert)
against the oracle.  Every token is checked up to T = 512 (small-batch
workload at T = 2..64, chunked prefill at T = 512 on both paths); at T = 4096
a seeded 512-token subset is (tokens are independent rows).  Token
permutation is checked at full size."""
import numpy as np
import pytest
import torch

import moe_synth
from tests._util import check_tokens, oracle_full, oracle_sampled, oracle_tokens, parity, min_rank_gap

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def m():
    import __graft_entry__
    __graft_entry__.build()
    import moe_decode_expert_gb300 as mod
    return mod


def _grouped(m, wl, g, T, out_dtype=None, ws=None, flags=0):
    cfg = m.cfg_from_workload(wl, out_dtype, flags)
    ids = torch.full((T, wl.top_k), -1, dtype=torch.int32, device=DEV)
    w = torch.full((T, wl.top_k), float("nan"), dtype=torch.float32, device=DEV)
    out = torch.full((T, wl.hidden), float("nan"), dtype=cfg.out_torch_dtype, device=DEV)
    if ws is None:
        ws = m.alloc_workspace(cfg, T, DEV)
    m.moe_grouped_forward(cfg, g["x"], g["router_w"], g["w13"], g["w2"], g["shared_w13"], g["shared_w2"],
                          g["shared_gate_w"], ids, w, out, ws)
    m.moe_query_status(ws)
    return ids, w, out


_REF = {}


def _ref_tokens(wl, layer, T, g, tokens):
    """Oracle rows for (workload, layer, T, tokens), computed once per module
    (both paths of a parametrised test see the same seeded inputs)."""
    key = (wl.name, layer, T, tuple(tokens))
    if key not in _REF:
        _REF[key] = oracle_tokens(wl, g, tokens)
    return _REF[key]


def _check_tokens(ids, w, out, ref, tokens, k):
    ok = 0
    for i, t in enumerate(tokens):
        if min_rank_gap(ref["logits"][i], k) > 1e-4:
            assert np.array_equal(ids[t].cpu().numpy(), ref["ids"][i]), t
            np.testing.assert_allclose(w[t].cpu().numpy(), ref["w"][i], rtol=1e-4, atol=1e-6)
            ok += 1
    parity(out[tokens], ref["out"])
    assert ok >= max(1, int(0.8 * len(tokens)))


SIMT, TC = 1, 2


@pytest.mark.parametrize("flags", [SIMT, TC], ids=["simt", "tcgen05"])
@pytest.mark.parametrize("T", [2, 4, 8, 16, 64])
def test_small_batch_zipf(m, T, flags):
    wl = moe_synth.workload("small_batch")
    g = moe_synth.make_layer(wl, 0, T, device=DEV)
    m.moe_reset_stats()
    ids, w, out = _grouped(m, wl, g, T, flags=flags)
    st = m.moe_get_stats()
    assert st["grouped_calls"] == 1 and st["grouped_tc_calls"] == (1 if flags == TC else 0)
    tokens = list(range(T))  # every token
    check_tokens(ids, w, out, _ref_tokens(wl, 0, T, g, tokens), tokens, wl.top_k)


@pytest.mark.parametrize("T", [9, 16, 17, 31, 32, 33])
def test_small_batch_fused_ranking_boundary(m, T):
    """Up to 32 tokens one single-CTA launch ranks (a warp per token), groups
    and lists the tiles; from 33 on the top-k launch also ranks each pair
    within its expert and one launch files the pairs, copies their x rows and
    lists the tiles.  Up to 16 tokens the W13 pass reads x itself (no gather
    launch).  Both sides of the boundaries, and ragged counts, match the
    oracle."""
    wl = moe_synth.workload("small_batch")
    g = moe_synth.make_layer(wl, 2, T, device=DEV)
    m.moe_reset_stats()
    ids, w, out = _grouped(m, wl, g, T, flags=TC)
    st = m.moe_get_stats()
    assert st["grouped_tc_calls"] == 1
    # router (+ top-k), ranking/grouping/tile lists (1) or filing/x rows/tile
    # lists (1), gather (1 for 17..32 tokens, and past 16384 pairs), W13, W2,
    # combine
    expect = (1 + 1 if T <= 32 else 2 + 1) + (1 if 16 < T <= 32 else 0) + 3
    assert st["kernels_launched"] == expect
    tokens = list(range(T))  # every token
    check_tokens(ids, w, out, _ref_tokens(wl, 2, T, g, tokens), tokens, wl.top_k)


@pytest.mark.parametrize("flags", [SIMT, TC], ids=["simt", "tcgen05"])
@pytest.mark.parametrize("T", [3, 65, 130])
def test_odd_token_counts_small_shapes(m, T, flags):
    wl = moe_synth.Workload("odd", 256, 32, 4, 64, 64, moe_synth.BF16, 1, 1.0, 0.05, 0.05, preset_id=6)
    d = moe_synth.make_layer(wl, 0, T)
    g = {k: (v.to(DEV) if v is not None else None) for k, v in d.items()}
    ids, w, out = _grouped(m, wl, g, T, out_dtype=3, flags=flags)
    ref = oracle_full(wl, d)
    gaps = min_rank_gap(ref["logits"], wl.top_k)
    good = gaps > 1e-5
    assert np.array_equal(ids.cpu().numpy()[good], ref["ids"][good])
    parity(out, ref["out"])


@pytest.mark.parametrize("flags", [SIMT, TC], ids=["simt", "tcgen05"])
def test_token_permutation_permutes_output(m, flags):
    wl = moe_synth.workload("small_batch")
    T = 16
    g = moe_synth.make_layer(wl, 1, T, device=DEV)
    _, _, out = _grouped(m, wl, g, T, flags=flags)
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(0)).to(DEV)
    g2 = dict(g)
    g2["x"] = g["x"][perm].contiguous()
    _, _, out2 = _grouped(m, wl, g2, T, flags=flags)
    assert torch.equal(out2, out[perm])


def test_ranked_grouping_repeats_on_one_workspace(m):
    """From 33 tokens the top-k launch ranks pairs with per-expert counters
    that a later launch of the same call zeroes again: calls repeated on one
    workspace, with a small batch in between, give the same bits."""
    wl = moe_synth.workload("small_batch")
    T = 100
    g = moe_synth.make_layer(wl, 8, T, device=DEV)
    g8 = moe_synth.make_layer(wl, 9, 8, device=DEV)
    cfg = m.cfg_from_workload(wl, None, TC)
    ws = m.alloc_workspace(cfg, T, DEV)
    first = _grouped(m, wl, g, T, flags=TC, ws=ws)
    tokens = list(range(0, T, 7))
    check_tokens(*first, _ref_tokens(wl, 8, T, g, tokens), tokens, wl.top_k)
    for _ in range(2):
        _grouped(m, wl, g8, 8, flags=TC, ws=ws)
        again = _grouped(m, wl, g, T, flags=TC, ws=ws)
        for a, b in zip(first, again):
            assert torch.equal(a, b)


@pytest.mark.parametrize("T", [4, 20, 64])
def test_tcgen05_path_fp16_sharded_shapes(m, T):
    """fp16 weights and tokens on the tcgen05 passes (kind::f16 with fp16
    operands, the activation split into two fp16 terms), every token against
    the oracle at the sharded shapes (I = 128, shared I = 128)."""
    wl = moe_synth.workload("sharded_decode")
    g = moe_synth.make_layer(wl, 4, T, device=DEV)
    m.moe_reset_stats()
    ids, w, out = _grouped(m, wl, g, T, flags=TC)
    assert m.moe_get_stats()["grouped_tc_calls"] == 1
    tokens = list(range(T))
    check_tokens(ids, w, out, oracle_tokens(wl, g, tokens), tokens, wl.top_k)


def test_grouped_t1_dispatches_to_decode_kernel(m):
    wl = moe_synth.workload("full_decode")
    g = moe_synth.make_layer(wl, 2, 1, device=DEV)
    m.moe_reset_stats()
    ids, w, out = _grouped(m, wl, g, 1)
    st = m.moe_get_stats()
    assert st["decode_fused_calls"] == 1 and st["grouped_calls"] == 0
    ref = oracle_sampled(wl, g, [0])
    _check_tokens(ids, w, out, ref, [0], wl.top_k)


@pytest.mark.parametrize("flags", [SIMT, TC], ids=["simt", "tcgen05"])
def test_chunked_prefill_512(m, flags):
    wl = moe_synth.workload("chunked_prefill")
    T = 512
    g = moe_synth.make_layer(wl, 0, T, device=DEV)
    ids, w, out = _grouped(m, wl, g, T, flags=flags)
    tokens = list(range(T))  # every token, at the full-width tile shapes
    check_tokens(ids, w, out, _ref_tokens(wl, 0, T, g, tokens), tokens, wl.top_k)


def test_chunked_prefill_4096_tcgen05(m):
    wl = moe_synth.workload("chunked_prefill")
    T = 4096
    g = moe_synth.make_layer(wl, 0, T, device=DEV)
    ids, w, out = _grouped(m, wl, g, T, flags=TC)
    # a seeded 512-token subset, plus the first and last token
    pick = np.random.default_rng(9).choice(np.arange(1, T - 1), 510, replace=False).tolist()
    tokens = sorted(set([0, T - 1] + pick))
    assert len(tokens) == 512
    check_tokens(ids, w, out, _ref_tokens(wl, 0, T, g, tokens), tokens, wl.top_k)


@pytest.mark.parametrize("T", [1023, 2049])
def test_chunked_prefill_ragged_token_counts(m, T):
    """Full prefill shapes at token counts with ragged tiles: 1023 (the router
    GEMM split into K parts, the x rows copied by the filing launch) and 2049
    (a gather launch): a seeded 128-token subset plus the first and last
    token."""
    wl = moe_synth.workload("chunked_prefill")
    g = moe_synth.make_layer(wl, 1, T, device=DEV)
    ids, w, out = _grouped(m, wl, g, T, flags=TC)
    pick = np.random.default_rng(T).choice(np.arange(1, T - 1), 128, replace=False).tolist()
    tokens = sorted(set([0, T - 1] + pick))
    check_tokens(ids, w, out, _ref_tokens(wl, 1, T, g, tokens), tokens, wl.top_k)


def test_simt_and_tcgen05_paths_agree(m):
    wl = moe_synth.workload("chunked_prefill")
    T = 300
    g = moe_synth.make_layer(wl, 1, T, device=DEV)
    i1, w1, o1 = _grouped(m, wl, g, T, out_dtype=3, flags=SIMT)
    i2, w2, o2 = _grouped(m, wl, g, T, out_dtype=3, flags=TC)
    assert torch.equal(i1, i2) and torch.equal(w1, w2)
    parity(o2, o1.double().cpu().numpy(), max_err_frac=1e-3, rel_l1=1e-4)


def test_graph_replays_after_a_smaller_call(m):
    """A CUDA graph captured at T = 16 still launches, with the same result,
    after an eager call at T = 2 on the same path (kernel shared-memory limits
    are raised, never lowered)."""
    wl = moe_synth.workload("small_batch")
    g16 = moe_synth.make_layer(wl, 3, 16, device=DEV)
    g2 = moe_synth.make_layer(wl, 4, 2, device=DEV)
    cfg = m.cfg_from_workload(wl, None, TC)
    ids = torch.empty(16, wl.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(16, wl.top_k, dtype=torch.float32, device=DEV)
    out = torch.empty(16, wl.hidden, dtype=cfg.out_torch_dtype, device=DEV)
    ws = m.alloc_workspace(cfg, 16, DEV)
    st = torch.cuda.Stream(device=DEV)
    st.wait_stream(torch.cuda.current_stream(DEV))

    def call():
        m.moe_grouped_forward(cfg, g16["x"], g16["router_w"], g16["w13"], g16["w2"], g16["shared_w13"],
                              g16["shared_w2"], g16["shared_gate_w"], ids, w, out, ws, st)

    with torch.cuda.stream(st):
        call()
    torch.cuda.synchronize()
    eager = out.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        call()
    _grouped(m, wl, g2, 2, flags=TC)  # a smaller call in between
    out.zero_()
    with torch.cuda.stream(st):
        graph.replay()
    torch.cuda.synchronize()
    m.moe_query_status(ws)
    assert torch.equal(out, eager)


@pytest.mark.parametrize("flags", [SIMT, TC], ids=["simt", "tcgen05"])
def test_residual_flag_grouped(m, flags):
    """MOE_FLAG_RESIDUAL on the T > 1 path: with fp32 output the result is
    exactly fl(block(x) + x) per element (the add follows the slot-order sum);
    with bf16 output it is that sum rounded once."""
    wl = moe_synth.workload("small_batch")
    T = 8
    g = moe_synth.make_layer(wl, 6, T, device=DEV)
    _, _, o0 = _grouped(m, wl, g, T, out_dtype=3, flags=flags)
    _, _, o1 = _grouped(m, wl, g, T, out_dtype=3, flags=flags | 8)
    assert torch.equal(o1, o0 + g["x"].float())
    _, _, o2 = _grouped(m, wl, g, T, flags=flags | 8)
    assert torch.equal(o2, o1.to(torch.bfloat16))


@pytest.mark.parametrize("flags", [SIMT, TC], ids=["simt", "tcgen05"])
@pytest.mark.parametrize("T", [24, 40])
def test_no_renormalisation_no_shared_expert(m, flags, T):
    """norm_topk = 0 (full-softmax weights) and no shared expert on both T > 1
    paths, every token against the oracle (T = 40: the ranked grouping, 64
    experts, top-6)."""
    wl = moe_synth.Workload("nonorm", 512, 64, 6, 128, 0, moe_synth.BF16, 0, 1.0, 0.05, 0.05, norm_topk=0,
                            preset_id=11)
    d = moe_synth.make_layer(wl, 0, T)
    g = {k_: (v.to(DEV) if v is not None else None) for k_, v in d.items()}
    ids, w, out = _grouped(m, wl, g, T, out_dtype=3, flags=flags)
    ref = oracle_full(wl, d)
    good = min_rank_gap(ref["logits"], wl.top_k) > 1e-4
    assert good.sum() >= T // 2
    assert np.array_equal(ids.cpu().numpy()[good], ref["ids"][good])
    np.testing.assert_allclose(w.cpu().numpy()[good], ref["w"][good], rtol=1e-4, atol=1e-7)
    assert np.all(w.sum(-1).cpu().numpy() < 1.0)  # full-softmax weights of k of E experts
    parity(out, ref["out"])


def test_fp16_batches_default_to_the_tensor_core_path(m):
    """fp16 batches run the tcgen05 passes by default from 4 tokens at these
    shapes (I = 128) and match the oracle on every token, as does an fp16
    batch of 6 on the CUDA-core kernels."""
    wl = moe_synth.workload("sharded_decode")
    T = 20
    g = moe_synth.make_layer(wl, 3, T, device=DEV)
    m.moe_reset_stats()
    ids, w, out = _grouped(m, wl, g, T)
    st = m.moe_get_stats()
    assert st["grouped_calls"] == 1 and st["grouped_tc_calls"] == 1 and st["kernels_launched"] > 1
    tokens = list(range(T))
    check_tokens(ids, w, out, oracle_tokens(wl, g, tokens), tokens, wl.top_k)
    T = 6
    g = moe_synth.make_layer(wl, 3, T, device=DEV)
    m.moe_reset_stats()
    ids, w, out = _grouped(m, wl, g, T, flags=SIMT)
    st = m.moe_get_stats()
    assert st["grouped_calls"] == 1 and st["grouped_tc_calls"] == 0
    tokens = list(range(T))
    check_tokens(ids, w, out, oracle_tokens(wl, g, tokens), tokens, wl.top_k)
    # at I = 128 the single launch is the default up to 3 tokens, the
    # tensor-core passes from 4
    for T, tc in ((3, 0), (4, 1)):
        g = moe_synth.make_layer(wl, 5, T, device=DEV)
        m.moe_reset_stats()
        ids, w, out = _grouped(m, wl, g, T)
        st = m.moe_get_stats()
        assert st["grouped_tc_calls"] == tc and (tc or st["kernels_launched"] == 1)
        tokens = list(range(T))
        check_tokens(ids, w, out, oracle_tokens(wl, g, tokens), tokens, wl.top_k)


def test_zero_tokens_is_a_no_op(m):
    wl = moe_synth.workload("small_batch")
    g = moe_synth.make_layer(wl, 0, 2, device=DEV)
    cfg = m.cfg_from_workload(wl)
    ws = m.alloc_workspace(cfg, 2, DEV)
    x0 = g["x"][:0]
    ids = torch.empty(0, wl.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(0, wl.top_k, dtype=torch.float32, device=DEV)
    out = torch.empty(0, wl.hidden, dtype=cfg.out_torch_dtype, device=DEV)
    m.moe_reset_stats()
    m.moe_grouped_forward(cfg, x0, g["router_w"], g["w13"], g["w2"], g["shared_w13"], g["shared_w2"],
                          g["shared_gate_w"], ids, w, out, ws)
    assert m.moe_get_stats()["kernels_launched"] == 0
