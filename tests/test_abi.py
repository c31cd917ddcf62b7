"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, sizes workspaces, and rejects bad arguments before touching
a GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m():
    import __graft_entry__
    __graft_entry__.build()
    import moe_decode_expert_gb300 as mod
    return mod


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("moe_router_topk", "moe_decode_forward", "moe_grouped_forward", "moe_workspace_bytes",
              "moe_last_error", "moe_query_status", "moe_get_stats"):
        assert n in names


def test_library_exports_every_declared_symbol(m):
    lib = m.library()
    for n in _declared():
        assert hasattr(lib, n), n
    assert set(_declared()) == set(m.EXPORTS)


def test_abi_version(m):
    assert m.moe_abi_version() == 2


def test_workspace_sizes(m):
    c = m.MoeCfg(2048, 256, 8, 128, 128, m.MOE_F16)
    one = m.moe_workspace_bytes(c, 1)
    assert one > 0 and one % 256 == 0
    # exchange words: (E + 1 padded) + (k*I + Is) words of 8 bytes, plus control and router logits
    assert one >= 256 + 258 * 8 + (1024 + 128) * 8
    many = m.moe_workspace_bytes(c, 64)
    P = 64 * 8 + 64
    assert many >= P * 2048 * 4 + P * 128 * 4
    assert m.moe_workspace_bytes(m.MoeCfg(2048, 256, 8, 127, 0, m.MOE_F16), 1) == 0  # I % 8 != 0


def _topk(m):
    return m.moe_topk_t(16, 16)


@pytest.mark.parametrize("field,value,code", [
    ("hidden", 0, 1), ("inter", 12, 2), ("top_k", 33, 2), ("top_k", 0, 1), ("dtype", 3, 2),
    ("n_experts", 2000, 2), ("flags", 32, 1), ("flags", 3, 1), ("flags", 17, 1), ("flags", 18, 1),
    ("norm_topk", 2, 1),
])
def test_bad_cfg_is_rejected_on_host(m, field, value, code):
    c = m.MoeCfg(256, 16, 2, 64, 0, m.MOE_F16).c()
    setattr(c, field, value)
    lib = m.library()
    vp = ctypes.c_void_p
    rc = lib.moe_decode_forward(ctypes.byref(c), vp(256), vp(512), vp(768), vp(1024), None, None, None,
                                _topk(m), vp(2048), vp(4096), 1 << 20, None)
    assert rc == code, m.moe_last_error()
    assert m.moe_last_error() != ""


def test_gate_without_shared_expert_is_invalid(m):
    c = m.MoeCfg(256, 16, 2, 64, 0, m.MOE_F16, has_shared_gate=1).c()
    rc = m.library().moe_router_topk(ctypes.byref(c), ctypes.c_void_p(256), ctypes.c_void_p(512), 1,
                                     _topk(m), None, ctypes.c_void_p(4096), 1 << 20, None)
    assert rc == 1


def test_unaligned_and_null_pointers(m):
    lib = m.library()
    c = m.MoeCfg(256, 16, 2, 64, 0, m.MOE_F16).c()
    vp = ctypes.c_void_p
    rc = lib.moe_decode_forward(ctypes.byref(c), vp(258), vp(512), vp(768), vp(1024), None, None, None,
                                _topk(m), vp(2048), vp(4096), 1 << 20, None)
    assert rc == 1 and "x" in m.moe_last_error()
    rc = lib.moe_decode_forward(ctypes.byref(c), vp(256), None, vp(768), vp(1024), None, None, None,
                                _topk(m), vp(2048), vp(4096), 1 << 20, None)
    assert rc == 1 and "router_w" in m.moe_last_error()
    # shared weights given although the cfg has no shared expert
    rc = lib.moe_decode_forward(ctypes.byref(c), vp(256), vp(512), vp(768), vp(1024), vp(1280), vp(1536), None,
                                _topk(m), vp(2048), vp(4096), 1 << 20, None)
    assert rc == 1


def test_small_or_misaligned_workspace(m):
    lib = m.library()
    cfg = m.MoeCfg(256, 16, 2, 64, 0, m.MOE_F16)
    c = cfg.c()
    vp = ctypes.c_void_p
    need = m.moe_workspace_bytes(cfg, 1)
    rc = lib.moe_decode_forward(ctypes.byref(c), vp(256), vp(512), vp(768), vp(1024), None, None, None,
                                _topk(m), vp(2048), vp(4096), need - 1, None)
    assert rc == 3
    rc = lib.moe_decode_forward(ctypes.byref(c), vp(256), vp(512), vp(768), vp(1024), None, None, None,
                                _topk(m), vp(2048), vp(4096 + 16), need, None)
    assert rc == 3
    rc = lib.moe_grouped_forward(ctypes.byref(c), vp(256), vp(512), vp(768), vp(1024), None, None, None,
                                 _topk(m), vp(2048), vp(4096), m.moe_workspace_bytes(cfg, 1), 4, None)
    assert rc == 3  # sized for T = 1, called with T = 4


def test_out_aliasing_x_is_rejected(m):
    lib = m.library()
    c = m.MoeCfg(256, 16, 2, 64, 0, m.MOE_F16).c()
    vp = ctypes.c_void_p
    rc = lib.moe_decode_forward(ctypes.byref(c), vp(256), vp(512), vp(768), vp(1024), None, None, None,
                                _topk(m), vp(256), vp(4096), 1 << 20, None)
    assert rc == 1


def test_zero_tokens_is_a_no_op(m):
    lib = m.library()
    c = m.MoeCfg(256, 16, 2, 64, 0, m.MOE_F16).c()
    vp = ctypes.c_void_p
    rc = lib.moe_grouped_forward(ctypes.byref(c), vp(256), vp(512), vp(768), vp(1024), None, None, None,
                                 _topk(m), vp(2048), None, 0, 0, None)
    assert rc == 0
    # with no tokens the per-token buffers may be NULL; the cfg is still checked
    rc = lib.moe_grouped_forward(ctypes.byref(c), None, vp(512), vp(768), vp(1024), None, None, None,
                                 m.moe_topk_t(None, None), None, None, 0, 0, None)
    assert rc == 0
    bad = m.MoeCfg(256, 16, 2, 60, 0, m.MOE_F16).c()
    rc = lib.moe_grouped_forward(ctypes.byref(bad), None, None, None, None, None, None, None,
                                 m.moe_topk_t(None, None), None, None, 0, 0, None)
    assert rc == 2
    rc = lib.moe_router_topk(ctypes.byref(c), None, None, 0, m.moe_topk_t(None, None), None, None, 0, None)
    assert rc == 0


def test_timeout_setting(m):
    with pytest.raises(m.MoeError):
        m.moe_set_wait_timeout_ns(10)
    m.moe_set_wait_timeout_ns(2_000_000_000)


def test_stats_roundtrip(m):
    m.moe_reset_stats()
    s = m.moe_get_stats()
    assert s == {"decode_fused_calls": 0, "router_calls": 0, "grouped_calls": 0, "grouped_tc_calls": 0,
                 "kernels_launched": 0, "decode_general_calls": 0}


def test_python_binding_checks_shapes(m):
    cfg = m.MoeCfg(256, 16, 2, 64, 0, m.MOE_F16)
    x = torch.zeros(1, 255, dtype=torch.float16)
    with pytest.raises(ValueError):
        m.moe_router_topk(cfg, x, torch.zeros(16, 256, dtype=torch.float16), torch.zeros(1, 2, dtype=torch.int32),
                          torch.zeros(1, 2), torch.zeros(16, dtype=torch.uint8))


def test_single_launch_batch_workspace(m):
    """2 <= T <= 8 on eligible shapes: the batch kernel's exchange words (16
    logit copies, activations and partial rows per (slot, token), slot T*k
    being the shared expert) are laid out; T = 9 has none of them."""
    c = m.MoeCfg(2048, 256, 8, 512, 512, m.MOE_BF16, has_shared_gate=1)
    for T in (2, 8):
        slots = T * 8 + 1
        words = 16 * T * 258 + slots * T * 512 + slots * T * 2048
        grouped_only = m.moe_workspace_bytes(m.MoeCfg(4096, 256, 8, 512, 512, m.MOE_BF16, has_shared_gate=1), T)
        assert m.moe_workspace_bytes(c, T) >= words * 8
        assert grouped_only > 0  # H = 4096: no batch regions, still a valid T > 1 workspace
    # the 16-token partial rows alone (129 slots x 16 tokens x 2048 words)
    # outweigh everything a 17-token workspace holds
    assert m.moe_workspace_bytes(c, 16) > m.moe_workspace_bytes(c, 17)


def test_tensor_core_path_workspace_is_laid_out_for_both_dtypes(m):
    bf = m.MoeCfg(2048, 256, 8, 512, 512, m.MOE_BF16, has_shared_gate=1)
    fp = m.MoeCfg(2048, 256, 8, 512, 512, m.MOE_F16, has_shared_gate=1)
    T = 512
    P = T * 8 + T
    assert m.moe_workspace_bytes(bf, T) == m.moe_workspace_bytes(fp, T)
    # fp32 activations and per-pair rows, gathered x rows and the two activation terms
    assert m.moe_workspace_bytes(bf, T) >= P * 512 * 4 + P * 2048 * 4 + P * 2048 * 2 + 2 * P * 512 * 2
