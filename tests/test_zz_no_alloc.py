"""The allocation-free decode entry point, through the C ABI.

Some callers cannot allocate device memory at all (a fixed pool reserved at
start-up, a plugin host that only hands over tensor pointers), so they cannot
provide the workspace moe_decode_forward needs.  moe_decode_forward_noalloc
keeps that scratch in a fixed array inside the library instead.  This test
calls it twice in a row and compares each result with moe_decode_forward on
the same inputs, within the tolerance the other parity tests use, and with the
oracle.  Its device status word lives in the same array; a wait that runs out
stays recorded there until moe_query_status(NULL) reads it."""
import ctypes

import numpy as np
import pytest
import torch

import moe_synth
from tests._util import _check_one_token, oracle_sampled, parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def m():
    import __graft_entry__
    __graft_entry__.build()
    import moe_decode_expert_gb300 as mod
    return mod


def _noalloc(m, cfg, g, ids, w, out):
    lib = m.library()
    c = cfg.c()
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = lib.moe_decode_forward_noalloc(ctypes.byref(c), p(g["x"]), p(g["router_w"]), p(g["w13"]), p(g["w2"]),
                                        p(g["shared_w13"]), p(g["shared_w2"]), p(g["shared_gate_w"]),
                                        m.moe_topk_t(ids.data_ptr(), w.data_ptr()), p(out),
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, m.moe_last_error()


@pytest.mark.parametrize("name", ["sharded_decode", "full_decode"])
def test_noalloc_matches_workspace_entry_two_calls(m, name):
    wl = moe_synth.workload(name)
    cfg = m.cfg_from_workload(wl)
    ws = m.alloc_workspace(cfg, 1, DEV)
    for layer in (0, 1):  # two calls in a row, different inputs
        g = moe_synth.make_layer(wl, layer, 1, device=DEV)
        ids0 = torch.empty(1, wl.top_k, dtype=torch.int32, device=DEV)
        w0 = torch.empty(1, wl.top_k, dtype=torch.float32, device=DEV)
        out0 = torch.empty(1, wl.hidden, dtype=cfg.out_torch_dtype, device=DEV)
        m.moe_decode_forward(cfg, g["x"], g["router_w"], g["w13"], g["w2"], g["shared_w13"], g["shared_w2"],
                             g["shared_gate_w"], ids0, w0, out0, ws)
        ids1 = torch.full_like(ids0, -1)
        w1 = torch.full_like(w0, float("nan"))
        out1 = torch.full_like(out0, float("nan"))
        _noalloc(m, cfg, g, ids1, w1, out1)
        torch.cuda.synchronize()
        m.moe_query_status(ws)
        assert torch.equal(ids0, ids1)
        np.testing.assert_allclose(w1.cpu().numpy(), w0.cpu().numpy(), rtol=1e-6)
        parity(out1, out0.double().cpu().numpy())
        _check_one_token(ids1, w1, out1, oracle_sampled(wl, g, [0]), wl.top_k)
    m.moe_query_status(None)  # no device-side error recorded in the built-in array


def test_noalloc_device_timeout_is_reported_and_later_calls_recover(m):
    """With a 1 us limit on every device wait, a full-width call almost surely
    has a CTA whose wait for the others runs out; the kernel records that in
    the array's status word and returns (no trap).  A later call with the
    normal limit computes the right result, leaves the recorded error in
    place, and moe_query_status(NULL) then reports and clears it."""
    wl = moe_synth.workload("full_decode")
    cfg = m.cfg_from_workload(wl)
    g = moe_synth.make_layer(wl, 3, 1, device=DEV)
    ref = oracle_sampled(wl, g, [0])
    ids = torch.empty(1, wl.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(1, wl.top_k, dtype=torch.float32, device=DEV)
    out = torch.empty(1, wl.hidden, dtype=cfg.out_torch_dtype, device=DEV)
    m.moe_query_status(None)
    seen = False
    for _ in range(20):
        try:
            m.moe_set_wait_timeout_ns(1000)
            _noalloc(m, cfg, g, ids, w, out)
        finally:
            m.moe_set_wait_timeout_ns(2_000_000_000)
        ids.fill_(-1)
        out.fill_(float("nan"))
        _noalloc(m, cfg, g, ids, w, out)  # normal limit: must be right
        torch.cuda.synchronize()
        _check_one_token(ids, w, out, ref, wl.top_k)
        try:
            m.moe_query_status(None)
        except m.MoeError as e:
            assert e.code == 5, e  # MOE_ERR_TIMEOUT, recorded by the 1 us call
            seen = True
            break
    assert seen, "no wait ran out in 20 calls with a 1 us limit"
    m.moe_query_status(None)  # read once, then clear


def test_noalloc_rejects_configs_beyond_its_scratch(m):
    big = m.MoeCfg(2048, 1024, 32, 4096, 4096, m.MOE_BF16)  # (E+1) + k*I + Is words exceed the array
    lib = m.library()
    c = big.c()
    vp = ctypes.c_void_p
    rc = lib.moe_decode_forward_noalloc(ctypes.byref(c), vp(256), vp(512), vp(768), vp(1024), vp(1280), vp(1536),
                                        None, m.moe_topk_t(16, 16), vp(2048), None)
    assert rc == 2 and "scratch" in m.moe_last_error()
