"""Reference oracle for the decode-step MoE block (ctypes front end).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the CPU
baseline leg of ``bench.py`` may import this module; the product path never
does.  The arithmetic lives in ``moe_oracle.cpp`` (single-threaded C++17,
IEEE double); this file only compiles it with g++, loads it and marshals
numpy arrays of raw fp16/bf16 bit patterns into it.

Restated from "BI-V100 inference work log" (kernel_worklog), Parts 1, 3, 4
and 10, and "Decode throughput analysis report", code-level profiling
section; see the header of ``moe_oracle.cpp`` for the readings taken.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")

F16 = 1
BF16 = 2


class _Cfg(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int32),
        ("n_experts", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("inter", ctypes.c_int32),
        ("shared_inter", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("norm_topk", ctypes.c_int32),
        ("has_shared_gate", ctypes.c_int32),
    ]


@dataclass(frozen=True)
class OracleCfg:
    hidden: int
    n_experts: int
    top_k: int
    inter: int
    shared_inter: int = 0
    dtype: int = F16          # F16 or BF16: the bytes of every input tensor
    norm_topk: int = 1
    has_shared_gate: int = 0

    def c(self) -> _Cfg:
        return _Cfg(self.hidden, self.n_experts, self.top_k, self.inter,
                    self.shared_inter, self.dtype, self.norm_topk, self.has_shared_gate)


def build(force: bool = False) -> str:
    """Compile the oracle shared library with g++ (no CUDA involved)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER
        u16p = P(ctypes.c_uint16)
        dp = P(ctypes.c_double)
        i32p = P(ctypes.c_int32)
        lib.oracle_decode.argtypes = [ctypes.c_uint16, ctypes.c_int32]
        lib.oracle_decode.restype = ctypes.c_double
        lib.oracle_router_token.argtypes = [P(_Cfg), u16p, u16p, dp, i32p, dp]
        lib.oracle_router_token.restype = ctypes.c_int
        lib.oracle_moe_forward.argtypes = [P(_Cfg), ctypes.c_int32, u16p, u16p,
                                           P(u16p), P(u16p), u16p, u16p, u16p,
                                           i32p, dp, dp, dp]
        lib.oracle_moe_forward.restype = ctypes.c_int
        lib.oracle_moe_forward_gather.argtypes = [P(_Cfg), ctypes.c_int32, u16p, u16p,
                                                  P(u16p), P(u16p), u16p, u16p, u16p, dp]
        lib.oracle_moe_forward_gather.restype = ctypes.c_int
        lib.oracle_w2_combine.argtypes = [P(_Cfg), dp, i32p, dp, P(u16p), dp]
        lib.oracle_w2_combine.restype = ctypes.c_int
        _lib = lib
    return _lib


def _u16(a):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bit patterns, got {a.dtype}")
    return a


def _ptr(a, ct):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ct))


def _expert_table(w, n_experts, per_expert_elems):
    """Build the E-entry pointer table the oracle takes for stacked expert weights.

    ``w`` is either one array [E, ...] or a dict {expert_id: array} holding only
    the experts that are present (the others stay NULL)."""
    keep = []
    table = (ctypes.POINTER(ctypes.c_uint16) * n_experts)()
    if isinstance(w, dict):
        for e, a in w.items():
            a = _u16(a)
            if a.size != per_expert_elems:
                raise ValueError("expert slice has the wrong size")
            keep.append(a)
            table[int(e)] = _ptr(a, ctypes.c_uint16)
    else:
        a = _u16(w)
        if a.size != n_experts * per_expert_elems:
            raise ValueError("stacked expert tensor has the wrong size")
        keep.append(a)
        base = a.ctypes.data
        for e in range(n_experts):
            table[e] = ctypes.cast(base + 2 * e * per_expert_elems, ctypes.POINTER(ctypes.c_uint16))
    return table, keep


def decode(bits: int, dtype: int) -> float:
    return _load().oracle_decode(int(bits), int(dtype))


def router(cfg: OracleCfg, x, wr):
    """One token: returns (logits[E] f64, ids[k] i32, w[k] f64)."""
    x, wr = _u16(x), _u16(wr)
    lg = np.zeros(cfg.n_experts, np.float64)
    ids = np.zeros(cfg.top_k, np.int32)
    w = np.zeros(cfg.top_k, np.float64)
    c = cfg.c()
    rc = _load().oracle_router_token(ctypes.byref(c), _ptr(x, ctypes.c_uint16), _ptr(wr, ctypes.c_uint16),
                                     _ptr(lg, ctypes.c_double), _ptr(ids, ctypes.c_int32),
                                     _ptr(w, ctypes.c_double))
    if rc:
        raise RuntimeError(f"oracle_router_token failed: {rc}")
    return lg, ids, w


def moe_forward(cfg: OracleCfg, x, wr, w13, w2, sw13=None, sw2=None, swg=None):
    """T tokens (x is [T, H] bits): returns dict(ids, w, logits, out) in fp64/int32."""
    x, wr = _u16(x), _u16(wr)
    T = x.size // cfg.hidden
    H, E, k, I = cfg.hidden, cfg.n_experts, cfg.top_k, cfg.inter
    t13, keep13 = _expert_table(w13, E, 2 * I * H)
    t2, keep2 = _expert_table(w2, E, H * I)
    sw13, sw2, swg = _u16(sw13), _u16(sw2), _u16(swg)
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    lg = np.zeros((T, E), np.float64)
    out = np.zeros((T, H), np.float64)
    c = cfg.c()
    rc = _load().oracle_moe_forward(ctypes.byref(c), T, _ptr(x, ctypes.c_uint16), _ptr(wr, ctypes.c_uint16),
                                    t13, t2, _ptr(sw13, ctypes.c_uint16), _ptr(sw2, ctypes.c_uint16),
                                    _ptr(swg, ctypes.c_uint16), _ptr(ids, ctypes.c_int32),
                                    _ptr(w, ctypes.c_double), _ptr(lg, ctypes.c_double),
                                    _ptr(out, ctypes.c_double))
    del keep13, keep2
    if rc:
        raise RuntimeError(f"oracle_moe_forward failed: {rc}")
    return {"ids": ids, "w": w, "logits": lg, "out": out}


def moe_forward_gather(cfg: OracleCfg, x, wr, w13, w2, sw13=None, sw2=None, swg=None):
    """Second formulation (copy-out of selected experts, dense, bmm, weighted sum)."""
    x, wr = _u16(x), _u16(wr)
    T = x.size // cfg.hidden
    H, E, I = cfg.hidden, cfg.n_experts, cfg.inter
    t13, keep13 = _expert_table(w13, E, 2 * I * H)
    t2, keep2 = _expert_table(w2, E, H * I)
    sw13, sw2, swg = _u16(sw13), _u16(sw2), _u16(swg)
    out = np.zeros((T, H), np.float64)
    c = cfg.c()
    rc = _load().oracle_moe_forward_gather(ctypes.byref(c), T, _ptr(x, ctypes.c_uint16),
                                           _ptr(wr, ctypes.c_uint16), t13, t2,
                                           _ptr(sw13, ctypes.c_uint16), _ptr(sw2, ctypes.c_uint16),
                                           _ptr(swg, ctypes.c_uint16), _ptr(out, ctypes.c_double))
    del keep13, keep2
    if rc:
        raise RuntimeError(f"oracle_moe_forward_gather failed: {rc}")
    return out


def w2_combine(cfg: OracleCfg, act, ids, w, w2):
    """Stage entry: out[h] = sum_j w[j] * sum_i W2[ids[j], h, i] * act[j, i]."""
    act = np.ascontiguousarray(act, np.float64)
    ids = np.ascontiguousarray(ids, np.int32)
    w = np.ascontiguousarray(w, np.float64)
    t2, keep2 = _expert_table(w2, cfg.n_experts, cfg.hidden * cfg.inter)
    out = np.zeros(cfg.hidden, np.float64)
    c = cfg.c()
    rc = _load().oracle_w2_combine(ctypes.byref(c), _ptr(act, ctypes.c_double), _ptr(ids, ctypes.c_int32),
                                   _ptr(w, ctypes.c_double), t2, _ptr(out, ctypes.c_double))
    del keep2
    if rc:
        raise RuntimeError(f"oracle_w2_combine failed: {rc}")
    return out
