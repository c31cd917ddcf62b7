"""Thin Python binding of the GB300 decode-step MoE library (``libmoe_gb300.so``).

The binding only marshals arguments: it takes torch tensors (device memory
and streams come from PyTorch), checks their shapes, dtypes and devices, and
passes raw pointers to the C ABI declared in ``include/moe.h``.  Every step
of the block runs in the library's CUDA kernels; there is no Python or CPU
fallback, and importing this package fails loudly if the library is missing.

Functions carry the C names (``moe_router_topk``, ``moe_decode_forward``,
``moe_grouped_forward``, ...); errors raise ``MoeError`` with the library's
``moe_last_error()`` text.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_F16, MOE_BF16, MOE_F32 = 1, 2, 3
_DT = {MOE_F16: torch.float16, MOE_BF16: torch.bfloat16, MOE_F32: torch.float32}
_DT_CODE = {torch.float16: MOE_F16, torch.bfloat16: MOE_BF16, torch.float32: MOE_F32}

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_DEVICE"}

# Every symbol include/moe.h declares.
EXPORTS = ("moe_abi_version", "moe_workspace_bytes", "moe_workspace_init", "moe_router_topk",
           "moe_decode_forward", "moe_grouped_forward", "moe_query_status", "moe_last_error",
           "moe_get_stats", "moe_reset_stats", "moe_set_wait_timeout_ns", "moe_test_wait_timeout",
           "moe_decode_forward_noalloc", "moe_sum_partials")


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{STATUS.get(code, code)}: {what}")
        self.code = code


class moe_cfg_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("hidden", "n_experts", "top_k", "inter", "shared_inter", "dtype",
                                              "out_dtype", "norm_topk", "has_shared_gate", "flags")]


class moe_topk_t(ctypes.Structure):
    _fields_ = [("ids", ctypes.c_void_p), ("weights", ctypes.c_void_p)]


class moe_stats_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("decode_fused_calls", "router_calls", "grouped_calls",
                                               "grouped_tc_calls", "kernels_launched", "decode_general_calls")]


MOE_FLAG_GROUPED_SIMT = 1
MOE_FLAG_GROUPED_TC = 2
MOE_FLAG_STATIC_WEIGHTS = 4
MOE_FLAG_RESIDUAL = 8
MOE_FLAG_GROUPED_SINGLE = 16


@dataclass(frozen=True)
class MoeCfg:
    hidden: int
    n_experts: int
    top_k: int
    inter: int
    shared_inter: int = 0
    dtype: int = MOE_BF16
    out_dtype: int | None = None
    norm_topk: int = 1
    has_shared_gate: int = 0
    flags: int = 0

    def c(self) -> moe_cfg_t:
        return moe_cfg_t(self.hidden, self.n_experts, self.top_k, self.inter, self.shared_inter, self.dtype,
                         self.dtype if self.out_dtype is None else self.out_dtype, self.norm_topk,
                         self.has_shared_gate, self.flags)

    @property
    def torch_dtype(self):
        return _DT[self.dtype]

    @property
    def out_torch_dtype(self):
        return _DT[self.dtype if self.out_dtype is None else self.out_dtype]


_lib = None


def use_library(path: str):
    """Load another build of this library (the phase-trace variant) instead of
    ``libmoe_gb300.so``; must come before the first call."""
    global LIB_PATH
    if _lib is not None:
        raise RuntimeError("the library is already loaded")
    LIB_PATH = path


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                          "(the MoE block has no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, u64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_uint64
    cfgp = ctypes.POINTER(moe_cfg_t)
    sig = {
        "moe_abi_version": ([], i32),
        "moe_workspace_bytes": ([cfgp, i32], sz),
        "moe_workspace_init": ([vp, sz, vp], ctypes.c_int),
        "moe_router_topk": ([cfgp, vp, vp, i32, moe_topk_t, vp, vp, sz, vp], ctypes.c_int),
        "moe_decode_forward": ([cfgp, vp, vp, vp, vp, vp, vp, vp, moe_topk_t, vp, vp, sz, vp], ctypes.c_int),
        "moe_grouped_forward": ([cfgp, vp, vp, vp, vp, vp, vp, vp, moe_topk_t, vp, vp, sz, i32, vp],
                                ctypes.c_int),
        "moe_query_status": ([vp, vp], ctypes.c_int),
        "moe_last_error": ([], ctypes.c_char_p),
        "moe_get_stats": ([ctypes.POINTER(moe_stats_t)], ctypes.c_int),
        "moe_reset_stats": ([], None),
        "moe_set_wait_timeout_ns": ([u64], ctypes.c_int),
        "moe_test_wait_timeout": ([vp, sz, vp], ctypes.c_int),
        "moe_decode_forward_noalloc": ([cfgp, vp, vp, vp, vp, vp, vp, vp, moe_topk_t, vp, vp], ctypes.c_int),
        "moe_sum_partials": ([vp, i32, ctypes.c_int64, vp, i32, vp, i32, vp], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def library():
    """The loaded ctypes library (raises if it was not built)."""
    return _load()


def _check(rc: int):
    if rc != 0:
        raise MoeError(rc, _load().moe_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t, name, shape, dtype, device):
    if t is None:
        raise ValueError(f"{name} is required")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ------------------------------------------------------------------ helpers
def moe_abi_version() -> int:
    return _load().moe_abi_version()


def moe_workspace_bytes(cfg: MoeCfg, T: int) -> int:
    c = cfg.c()
    return int(_load().moe_workspace_bytes(ctypes.byref(c), int(T)))


def alloc_workspace(cfg: MoeCfg, T: int, device) -> torch.Tensor:
    """A zero-filled, 256-byte aligned workspace for up to T tokens of cfg."""
    n = moe_workspace_bytes(cfg, T)
    if n == 0:
        raise MoeError(1, "invalid cfg")
    ws = torch.zeros(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    return ws[off:off + n]


def moe_workspace_init(ws: torch.Tensor, stream=None):
    _check(_load().moe_workspace_init(_ptr(ws), ws.numel(), _stream(stream)))


def moe_query_status(ws: torch.Tensor | None, stream=None):
    """Synchronise the stream, then read and clear the device status word of
    ``ws`` (None: the built-in array of moe_decode_forward_noalloc)."""
    _check(_load().moe_query_status(_ptr(ws), _stream(stream)))


def moe_last_error() -> str:
    return _load().moe_last_error().decode(errors="replace")


def moe_get_stats() -> dict:
    s = moe_stats_t()
    _check(_load().moe_get_stats(ctypes.byref(s)))
    return {n: int(getattr(s, n)) for n, _ in moe_stats_t._fields_}


def moe_reset_stats():
    _load().moe_reset_stats()


def moe_set_wait_timeout_ns(ns: int):
    _check(_load().moe_set_wait_timeout_ns(int(ns)))


def moe_test_wait_timeout(ws: torch.Tensor, stream=None):
    _check(_load().moe_test_wait_timeout(_ptr(ws), ws.numel(), _stream(stream)))


# --------------------------------------------------------------- the block
def moe_router_topk(cfg: MoeCfg, x, router_w, ids, weights, ws, logits=None, stream=None):
    """Router logits, softmax and top-k for x [T, H]; fills ids/weights [T, k]."""
    T = x.shape[0]
    dev = x.device
    dt = cfg.torch_dtype
    _need(x, "x", (T, cfg.hidden), dt, dev)
    _need(router_w, "router_w", (cfg.n_experts, cfg.hidden), dt, dev)
    _need(ids, "ids", (T, cfg.top_k), torch.int32, dev)
    _need(weights, "weights", (T, cfg.top_k), torch.float32, dev)
    if logits is not None:
        _need(logits, "logits", (T, cfg.n_experts), torch.float32, dev)
    c = cfg.c()
    _check(_load().moe_router_topk(ctypes.byref(c), _ptr(x), _ptr(router_w), T,
                                   moe_topk_t(ids.data_ptr(), weights.data_ptr()), _ptr(logits),
                                   _ptr(ws), ws.numel(), _stream(stream)))


def _block_args(cfg, x, router_w, w13, w2, shared_w13, shared_w2, shared_gate_w, ids, weights, out, T):
    dev = x.device
    dt = cfg.torch_dtype
    H, E, k, I, Is = cfg.hidden, cfg.n_experts, cfg.top_k, cfg.inter, cfg.shared_inter
    _need(x, "x", (T, H), dt, dev)
    _need(router_w, "router_w", (E, H), dt, dev)
    _need(w13, "w13", (E, 2 * I, H), dt, dev)
    _need(w2, "w2", (E, H, I), dt, dev)
    if Is:
        _need(shared_w13, "shared_w13", (2 * Is, H), dt, dev)
        _need(shared_w2, "shared_w2", (H, Is), dt, dev)
    if cfg.has_shared_gate:
        _need(shared_gate_w, "shared_gate_w", (H,), dt, dev)
    _need(ids, "ids", (T, k), torch.int32, dev)
    _need(weights, "weights", (T, k), torch.float32, dev)
    _need(out, "out", (T, H), cfg.out_torch_dtype, dev)
    return (_ptr(x), _ptr(router_w), _ptr(w13), _ptr(w2), _ptr(shared_w13), _ptr(shared_w2),
            _ptr(shared_gate_w), moe_topk_t(ids.data_ptr(), weights.data_ptr()), _ptr(out))


def moe_decode_forward(cfg: MoeCfg, x, router_w, w13, w2, shared_w13, shared_w2, shared_gate_w, ids, weights,
                       out, ws, stream=None):
    """One decode token (x [1, H]) through the whole block in one kernel launch."""
    args = _block_args(cfg, x, router_w, w13, w2, shared_w13, shared_w2, shared_gate_w, ids, weights, out, 1)
    c = cfg.c()
    _check(_load().moe_decode_forward(ctypes.byref(c), *args, _ptr(ws), ws.numel(), _stream(stream)))


def moe_decode_forward_noalloc(cfg: MoeCfg, x, router_w, w13, w2, shared_w13, shared_w2, shared_gate_w, ids,
                               weights, out, stream=None):
    """moe_decode_forward for callers that cannot allocate a workspace: the
    scratch is a fixed array inside the library (see include/moe.h)."""
    args = _block_args(cfg, x, router_w, w13, w2, shared_w13, shared_w2, shared_gate_w, ids, weights, out, 1)
    c = cfg.c()
    _check(_load().moe_decode_forward_noalloc(ctypes.byref(c), *args, _stream(stream)))


def moe_grouped_forward(cfg: MoeCfg, x, router_w, w13, w2, shared_w13, shared_w2, shared_gate_w, ids, weights,
                        out, ws, stream=None):
    """T tokens (x [T, H]) through the block; T > 1 groups (token, expert) pairs by expert."""
    T = x.shape[0]
    args = _block_args(cfg, x, router_w, w13, w2, shared_w13, shared_w2, shared_gate_w, ids, weights, out, T)
    c = cfg.c()
    _check(_load().moe_grouped_forward(ctypes.byref(c), *args, _ptr(ws), ws.numel(), T, _stream(stream)))


def moe_sum_partials(partials, out, residual=None, stream=None):
    """out = sum over dim 0 of fp32 ``partials`` [n_parts, ...] (+ residual),
    rounded once to out's dtype; the sum runs in part order."""
    if partials.dtype != torch.float32 or not partials.is_contiguous():
        raise ValueError("partials must be contiguous fp32")
    n = out.numel()
    if partials.numel() != partials.shape[0] * n or not out.is_contiguous():
        raise ValueError("partials must be [n_parts, *out.shape], out contiguous")
    if out.device != partials.device:
        raise ValueError("partials and out must be on one device")
    rdt = 0
    if residual is not None:
        if residual.numel() != n or not residual.is_contiguous() or residual.dtype not in (torch.float16,
                                                                                           torch.bfloat16):
            raise ValueError("residual must be a contiguous fp16/bf16 tensor shaped like out")
        rdt = _DT_CODE[residual.dtype]
    _check(_load().moe_sum_partials(_ptr(partials), partials.shape[0], n, _ptr(residual), rdt, _ptr(out),
                                    _DT_CODE[out.dtype], _stream(stream)))


def cfg_from_workload(wl, out_dtype=None, flags=0) -> MoeCfg:
    """MoeCfg for a synthetic workload description (moe_synth.Workload)."""
    return MoeCfg(wl.hidden, wl.n_experts, wl.top_k, wl.inter, wl.shared_inter, wl.dtype, out_dtype,
                  wl.norm_topk, wl.has_shared_gate, flags)
