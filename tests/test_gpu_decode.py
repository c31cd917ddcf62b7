"""GPU parity of the single-launch T = 1 decode kernel against the fp64 oracle,
through the C ABI.  Ids must match bit for bit; outputs within
max|err| <= 1e-2 max|ref| and relative L1 <= 2e-3."""
import math

import numpy as np
import pytest
import torch

import moe_synth
from tests._util import oracle_full, oracle_sampled, parity, min_rank_gap

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def m():
    import __graft_entry__
    __graft_entry__.build()
    import moe_decode_expert_gb300 as mod
    mod.moe_set_wait_timeout_ns(2_000_000_000)
    return mod


def _to(d, dev=DEV):
    return {k: (v.to(dev) if v is not None else None) for k, v in d.items()}


def _decode(m, wl, g, out_dtype=None, ws=None, flags=0):
    cfg = m.cfg_from_workload(wl, out_dtype, flags)
    ids = torch.full((1, wl.top_k), -1, dtype=torch.int32, device=DEV)
    w = torch.full((1, wl.top_k), float("nan"), dtype=torch.float32, device=DEV)
    out = torch.full((1, wl.hidden), float("nan"), dtype=cfg.out_torch_dtype, device=DEV)
    if ws is None:
        ws = m.alloc_workspace(cfg, 1, DEV)
    m.moe_decode_forward(cfg, g["x"], g["router_w"], g["w13"], g["w2"], g["shared_w13"], g["shared_w2"],
                         g["shared_gate_w"], ids, w, out, ws)
    m.moe_query_status(ws)
    return ids, w, out


def test_library_is_the_native_path(m):
    m.moe_reset_stats()
    wl = moe_synth.workload("tiny")
    _decode(m, wl, _to(moe_synth.make_layer(wl, 0, 1)))
    st = m.moe_get_stats()
    assert st["decode_fused_calls"] == 1 and st["kernels_launched"] == 1
    assert st["decode_general_calls"] == 0  # a standard shape: the specialised kernel
    maps = open("/proc/self/maps").read()
    assert "libmoe_gb300.so" in maps


@pytest.mark.parametrize("out_dtype", [3, None])
def test_tiny_config(m, out_dtype):
    wl = moe_synth.workload("tiny")
    for layer in range(4):
        d = moe_synth.make_layer(wl, layer, 1)
        ref = oracle_full(wl, d)
        ids, w, out = _decode(m, wl, _to(d), out_dtype)
        assert min_rank_gap(ref["logits"], wl.top_k)[0] > 1e-5
        assert np.array_equal(ids.cpu().numpy(), ref["ids"])
        np.testing.assert_allclose(w.cpu().numpy(), ref["w"], rtol=1e-5, atol=1e-7)
        if out_dtype == 3:
            parity(out, ref["out"])
        else:
            # fp16 output of tiny values sits in the subnormal range: compare with the
            # oracle rounded to fp16 (round to nearest even), within one unit there.
            ref16 = torch.from_numpy(ref["out"]).to(torch.float16).double().numpy()
            got = out.cpu().double().numpy()
            ulp = np.maximum(np.abs(np.spacing(ref16.astype(np.float16))).astype(np.float64), 2.0 ** -24)
            assert np.all(np.abs(got - ref16) <= ulp + 1e-12)


@pytest.mark.parametrize("flags", [0, 4], ids=["plain", "static_weights"])
@pytest.mark.parametrize("name", ["sharded_decode", "full_decode"])
def test_full_size_layers(m, name, flags):
    wl = moe_synth.workload(name)
    ws = m.alloc_workspace(m.cfg_from_workload(wl), 1, DEV)
    for layer in (0, 17, 35):
        g = moe_synth.make_layer(wl, layer, 1, device=DEV)
        ids, w, out = _decode(m, wl, g, ws=ws, flags=flags)
        ref = oracle_sampled(wl, g, [0])
        assert min_rank_gap(ref["logits"], wl.top_k)[0] > 1e-4
        assert np.array_equal(ids.cpu().numpy(), ref["ids"])
        np.testing.assert_allclose(w.cpu().numpy(), ref["w"], rtol=1e-4, atol=1e-6)
        parity(out, ref["out"])
        del g


def _closed_form_layer(wl, c, cs, gate_zero=True):
    H, E, I, Is = wl.hidden, wl.n_experts, wl.inter, wl.shared_inter
    dt = wl.torch_dtype
    d = {"x": torch.ones(1, H, dtype=dt),
         "router_w": (torch.randn(E, H, generator=torch.Generator().manual_seed(3)) * 0.02).to(dt)}
    w13 = torch.empty(E, 2 * I, H, dtype=dt)
    w13[:, :I] = c / H
    w13[:, I:] = 1.0 / H
    d["w13"] = w13
    d["w2"] = torch.ones(E, H, I, dtype=dt)
    if Is:
        s13 = torch.empty(2 * Is, H, dtype=dt)
        s13[:Is] = cs / H
        s13[Is:] = 1.0 / H
        d["shared_w13"] = s13
        d["shared_w2"] = torch.ones(H, Is, dtype=dt)
    else:
        d["shared_w13"] = d["shared_w2"] = None
    d["shared_gate_w"] = torch.zeros(H, dtype=dt) if wl.has_shared_gate else None
    return d


@pytest.mark.parametrize("name", ["sharded_decode", "full_decode"])
def test_closed_form(m, name):
    """x = 1, gate rows c/H, up rows 1/H, W2 = 1: out = I*silu(c) + g*Is*silu(cs)."""
    wl = moe_synth.workload(name)
    c, cs = 4.0, 2.0
    d = _closed_form_layer(wl, c, cs)
    silu = lambda v: v / (1.0 + math.exp(-v))
    expect = wl.inter * silu(c) + (0.5 if wl.has_shared_gate else 1.0) * wl.shared_inter * silu(cs)
    _, w, out = _decode(m, wl, _to(d), out_dtype=3)
    assert abs(w.sum().item() - 1.0) < 1e-6
    np.testing.assert_allclose(out.cpu().double().numpy(), expect, rtol=2e-6)


@pytest.mark.parametrize("out_dtype", [3, None])
def test_known_data_128(m, out_dtype):
    """The work log's known-data check through the whole block: x = 1 and a zero
    router make every logit 0 (ids 0..7, weights 1/8); gate rows 64/H and up
    rows 2^-6/H make every activation exactly 1; W2 = 1 gives 128.0 per output."""
    wl = moe_synth.workload("sharded_decode")
    H, E, I = wl.hidden, wl.n_experts, wl.inter
    dt = wl.torch_dtype
    d = {"x": torch.ones(1, H, dtype=dt), "router_w": torch.zeros(E, H, dtype=dt)}
    w13 = torch.empty(E, 2 * I, H, dtype=dt)
    w13[:, :I] = 64.0 / H
    w13[:, I:] = 2.0 ** -6 / H
    d["w13"] = w13
    d["w2"] = torch.ones(E, H, I, dtype=dt)
    d["shared_w13"] = torch.ones(2 * wl.shared_inter, H, dtype=dt) / H
    d["shared_w2"] = torch.zeros(H, wl.shared_inter, dtype=dt)
    d["shared_gate_w"] = None
    ids, w, out = _decode(m, wl, _to(d), out_dtype)
    assert ids.cpu().tolist() == [list(range(8))]
    assert torch.all(w == 0.125)
    assert torch.all(out.float() == 128.0), out.float().unique()


def test_zero_input_all_ties(m):
    wl = moe_synth.workload("full_decode")
    g = moe_synth.make_layer(wl, 0, 1, device=DEV)
    g["x"] = torch.zeros_like(g["x"])
    ids, w, out = _decode(m, wl, g)
    assert ids.cpu().tolist() == [list(range(wl.top_k))]
    assert torch.all(w == 1.0 / wl.top_k)
    assert torch.all(out.float() == 0)


def test_duplicated_router_rows_rank_lower_index_first(m):
    wl = moe_synth.workload("sharded_decode")
    g = moe_synth.make_layer(wl, 1, 1, device=DEV)
    top = (g["x"][0].float() * 0.05).to(g["x"].dtype)
    for e in (200, 3, 77):
        g["router_w"][e] = top
    ids, w, _ = _decode(m, wl, g)
    assert ids.cpu().tolist()[0][:3] == [3, 77, 200]
    assert w[0, 0] == w[0, 1] == w[0, 2]


@pytest.mark.parametrize("E,k,I,Is,gate,dt,norm", [
    (32, 4, 64, 64, 1, moe_synth.BF16, 1),
    (512, 8, 32, 0, 0, moe_synth.F16, 1),
    (64, 6, 48, 16, 0, moe_synth.BF16, 0),
    (1024, 32, 16, 8, 1, moe_synth.F16, 1),
    (320, 8, 200, 64, 1, moe_synth.BF16, 1),  # two pairs in flight per warp, general ranking and combine
])
def test_shape_variants(m, E, k, I, Is, gate, dt, norm):
    wl = moe_synth.Workload("v", 512, E, k, I, Is, dt, gate, 1.0, 0.05, 0.05, norm_topk=norm, preset_id=9)
    # the launch takes the specialised kernel only for the standard shapes
    H = 512
    G = min(torch.cuda.get_device_properties(0).multi_processor_count, k * I)
    standard = E <= 256 and k <= 8 and H >= G and -(-H // G) <= 16 and I % 16 == 0 and Is % 16 == 0
    m.moe_reset_stats()
    calls = 0
    for layer in range(2):
        d = moe_synth.make_layer(wl, layer, 1)
        ref = oracle_full(wl, d)
        if min_rank_gap(ref["logits"], k)[0] < 1e-5:
            continue
        ids, w, out = _decode(m, wl, _to(d), out_dtype=3)
        calls += 1
        assert np.array_equal(ids.cpu().numpy(), ref["ids"])
        np.testing.assert_allclose(w.cpu().numpy(), ref["w"], rtol=1e-5, atol=1e-7)
        parity(out, ref["out"])
    assert m.moe_get_stats()["decode_general_calls"] == (0 if standard else calls)


def test_repeated_calls_share_one_workspace(m):
    """The launch epoch advances every call; stale exchange words of earlier
    calls (and of another cfg's layout) must never be taken for fresh ones."""
    wl = moe_synth.workload("tiny")
    wl2 = moe_synth.Workload("v2", 256, 32, 4, 64, 32, moe_synth.F16, 1, 1.0, 0.05, 0.05, preset_id=8)
    ws = m.alloc_workspace(m.cfg_from_workload(wl2), 1, DEV)
    d1 = moe_synth.make_layer(wl, 0, 1)
    d2 = moe_synth.make_layer(wl2, 0, 1)
    g1, g2 = _to(d1), _to(d2)
    r1, r2 = oracle_full(wl, d1), oracle_full(wl2, d2)
    for it in range(40):
        wl_i, g, r = (wl, g1, r1) if it % 3 else (wl2, g2, r2)
        ids, _, out = _decode(m, wl_i, g, out_dtype=3, ws=ws)
        assert np.array_equal(ids.cpu().numpy(), r["ids"])
        parity(out, r["out"])


@pytest.mark.parametrize("flags", [0, 4], ids=["plain", "static_weights"])
def test_cuda_graph_of_layers(m, flags):
    """Rotated layers captured in one CUDA graph and replayed: equal to eager."""
    wl = moe_synth.workload("sharded_decode")
    cfg = m.cfg_from_workload(wl, None, flags)
    L = 4
    layers = [moe_synth.make_layer(wl, l, 1, device=DEV) for l in range(L)]
    ws = m.alloc_workspace(cfg, 1, DEV)
    outs = [torch.empty(1, wl.hidden, dtype=cfg.out_torch_dtype, device=DEV) for _ in range(L)]
    ids = [torch.empty(1, wl.top_k, dtype=torch.int32, device=DEV) for _ in range(L)]
    ws_ = [torch.empty(1, wl.top_k, dtype=torch.float32, device=DEV) for _ in range(L)]

    def step():
        for l, g in enumerate(layers):
            m.moe_decode_forward(cfg, g["x"], g["router_w"], g["w13"], g["w2"], g["shared_w13"], g["shared_w2"],
                                 g["shared_gate_w"], ids[l], ws_[l], outs[l], ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())  # the layers were generated on the default stream
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    for o in outs:
        o.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    m.moe_query_status(ws)
    for a, b in zip(eager, outs):
        assert torch.equal(a, b)


def test_timeout_path_records_and_recovers(m):
    """A wait on a flag nothing sets gives up after the limit, records
    MOE_ERR_TIMEOUT, and leaves the context usable."""
    wl = moe_synth.workload("tiny")
    cfg = m.cfg_from_workload(wl)
    ws = m.alloc_workspace(cfg, 1, DEV)
    m.moe_set_wait_timeout_ns(2_000_000)
    try:
        m.moe_test_wait_timeout(ws)
        with pytest.raises(m.MoeError) as ei:
            m.moe_query_status(ws)
        assert ei.value.code == 5
        assert "test wait" in str(ei.value)
    finally:
        m.moe_set_wait_timeout_ns(2_000_000_000)
    m.moe_workspace_init(ws)
    d = moe_synth.make_layer(wl, 0, 1)
    ids, _, out = _decode(m, wl, _to(d), out_dtype=3, ws=ws)
    ref = oracle_full(wl, d)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    parity(out, ref["out"])


@pytest.mark.parametrize("flags", [0, 4], ids=["plain", "static_weights"])
def test_chained_layers_read_the_previous_output(m, flags):
    """Each layer's x is the previous layer's out, written by the previous kernel
    on the stream.  A layer kernel launches early (programmatic dependent launch;
    with static weights it also streams weights and prefetches x into L2 before
    its wait) but must read x only after the previous layer has completed.
    Eager and graph-replayed chains agree bit for bit, and every layer matches the
    oracle run on the input the GPU actually used."""
    wl = moe_synth.workload("sharded_decode")  # fp16 in and out, so out can feed the next layer
    cfg = m.cfg_from_workload(wl, None, flags)
    L = 4
    layers = []
    for l in range(L):
        g = moe_synth.make_layer(wl, l, 1, device=DEV, weights_only=True)
        # larger down projections keep the chained activations near unit scale
        g["w2"] = (g["w2"].float() * 8).to(g["w2"].dtype)
        g["shared_w2"] = (g["shared_w2"].float() * 8).to(g["shared_w2"].dtype)
        layers.append(g)
    bufs = [moe_synth.make_x(wl, 0, 1, DEV)] + [torch.empty(1, wl.hidden, dtype=wl.torch_dtype, device=DEV)
                                                for _ in range(L)]
    ids = [torch.empty(1, wl.top_k, dtype=torch.int32, device=DEV) for _ in range(L)]
    wts = [torch.empty(1, wl.top_k, dtype=torch.float32, device=DEV) for _ in range(L)]
    ws = m.alloc_workspace(cfg, 1, DEV)

    def step():
        for l, g in enumerate(layers):
            m.moe_decode_forward(cfg, bufs[l], g["router_w"], g["w13"], g["w2"], g["shared_w13"], g["shared_w2"],
                                 g["shared_gate_w"], ids[l], wts[l], bufs[l + 1], ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    m.moe_query_status(ws)
    for l, g in enumerate(layers):
        ref = oracle_sampled(wl, {**g, "x": bufs[l]}, [0])
        lg = ref["logits"]
        if min_rank_gap(lg, wl.top_k)[0] > 1e-4 * np.abs(lg).max():
            assert np.array_equal(ids[l].cpu().numpy(), ref["ids"])
        parity(bufs[l + 1], ref["out"])
        assert 0.05 < bufs[l + 1].float().abs().max().item() < 1e3
    eager = [b.clone() for b in bufs[1:]]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    for b in bufs[1:]:
        b.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    m.moe_query_status(ws)
    for a, b in zip(eager, bufs[1:]):
        assert torch.equal(a, b)


def _ulp(v, dt):
    """Spacing of the storage type (fp16 / bf16) at |v| (normal range; the
    subnormal spacing below it)."""
    mant, emin = (10, -14) if dt == torch.float16 else (7, -126)
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** emin)))
    return 2.0 ** (e - mant)


@pytest.mark.parametrize("name,flags", [("full_decode", 8 | 4), ("sharded_decode", 8)],
                         ids=["full_width_static", "sharded"])
def test_residual_chain_layers(m, name, flags):
    """h <- h + MoE_l(h) over 4 layers, the residual add fused into the output
    write (MOE_FLAG_RESIDUAL): each layer reads the previous layer's output.
    Every layer is checked against x_l + oracle(x_l) on the input x_l the GPU
    actually used: within the tolerance, and elementwise within half a
    storage-type ulp of that sum plus 1e-3 of the block's own output scale.
    Eager and graph-replayed chains agree bit for bit."""
    wl = moe_synth.workload(name)
    cfg = m.cfg_from_workload(wl, None, flags)
    L = 4
    layers = [moe_synth.make_layer(wl, l + 5, 1, device=DEV, weights_only=True) for l in range(L)]
    bufs = [moe_synth.make_x(wl, 5, 1, DEV)] + [torch.empty(1, wl.hidden, dtype=wl.torch_dtype, device=DEV)
                                                for _ in range(L)]
    ids = [torch.empty(1, wl.top_k, dtype=torch.int32, device=DEV) for _ in range(L)]
    wts = [torch.empty(1, wl.top_k, dtype=torch.float32, device=DEV) for _ in range(L)]
    ws = m.alloc_workspace(cfg, 1, DEV)

    def step():
        for l, g in enumerate(layers):
            m.moe_decode_forward(cfg, bufs[l], g["router_w"], g["w13"], g["w2"], g["shared_w13"], g["shared_w2"],
                                 g["shared_gate_w"], ids[l], wts[l], bufs[l + 1], ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    m.moe_query_status(ws)
    for l, g in enumerate(layers):
        ref = oracle_sampled(wl, {**g, "x": bufs[l]}, [0])
        xl = bufs[l].double().cpu().numpy()
        exact = xl + ref["out"]
        got = bufs[l + 1].double().cpu().numpy()
        if min_rank_gap(ref["logits"], wl.top_k)[0] > 1e-4:
            assert np.array_equal(ids[l].cpu().numpy(), ref["ids"])
        parity(bufs[l + 1], exact)
        bound = 0.5 * _ulp(exact, wl.torch_dtype) + 1e-3 * np.abs(ref["out"]).max()
        assert np.all(np.abs(got - exact) <= bound), np.abs(got - exact).max()
    eager = [b.clone() for b in bufs[1:]]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    for b in bufs[1:]:
        b.zero_()
    graph.replay()
    torch.cuda.synchronize()
    m.moe_query_status(ws)
    for a, b in zip(eager, bufs[1:]):
        assert torch.equal(a, b)


def test_residual_flag_adds_x_after_the_block(m):
    """With fp32 output the residual result is exactly fl(block(x) + x): the
    add comes after the block's own sum, on x decoded exactly."""
    wl = moe_synth.workload("full_decode")
    g = moe_synth.make_layer(wl, 7, 1, device=DEV)
    outs = []
    for flags in (0, 8):
        cfg = m.cfg_from_workload(wl, 3, flags)
        ids = torch.empty(1, wl.top_k, dtype=torch.int32, device=DEV)
        w = torch.empty(1, wl.top_k, dtype=torch.float32, device=DEV)
        out = torch.empty(1, wl.hidden, dtype=torch.float32, device=DEV)
        ws = m.alloc_workspace(cfg, 1, DEV)
        m.moe_decode_forward(cfg, g["x"], g["router_w"], g["w13"], g["w2"], g["shared_w13"], g["shared_w2"],
                             g["shared_gate_w"], ids, w, out, ws)
        m.moe_query_status(ws)
        outs.append(out)
    assert torch.equal(outs[1], outs[0] + g["x"].float())
