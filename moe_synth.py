"""Seeded synthetic inputs for the decode-step MoE block.

This module is shared by the tests, the benchmark and the oracle side.  It
holds none of the block's arithmetic: it only draws seeded normal numbers,
rounds them to the storage dtype, and builds the structured inputs the
workloads call for (a Zipf-biased router, exactly representable weights for
closed-form checks).  Tensors are returned as torch tensors in fp16/bf16 on
the requested device; ``bits()`` gives the raw uint16 patterns the oracle
reads.

Workloads (shapes of the pages' model, Qwen3-style 256-expert top-8 MoE):

* ``tiny``            H=256, E=16, k=2, I=64, no shared expert, fp16, T=1,
                      x, W13, W2 ~ N(0, 0.02), router ~ N(0, 0.1), 1 layer.
* ``sharded_decode``  H=2048, E=256, k=8, I=128, shared I=128, fp16, T=1,
                      weights ~ N(0, 0.02), x ~ N(0, 1), 36 layers.  One TP=4
                      shard of the model ("BI-V100 inference work log",
                      Parts 2-3 and 10: W13 256x2048 and W2 2048x128 per expert).
* ``full_decode``     H=2048, E=256, k=8, I=512, shared I=512 with a sigmoid
                      gate, bf16, weights ~ N(0, 0.02), x ~ N(0, 1), T=1,
                      36 layers (~58 GB).
* ``small_batch``     full_decode shapes, T in {2, 4, 8, 16, 64}; column 0 of
                      x is 1 and column 0 of the router is -1.1*ln(rank_e)
                      (rank_e a seeded permutation of 1..E), so expert
                      popularity follows Zipf(s=1.1).
* ``chunked_prefill`` full_decode shapes, T in {512, 4096}, router
                      ~ N(0, 1/sqrt(H)) so logits ~ N(0, 1), 4 layers.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

F16, BF16, F32 = 1, 2, 3          # same codes as the library's dtype enum
_TORCH_DT = {F16: torch.float16, BF16: torch.bfloat16, F32: torch.float32}


@dataclass(frozen=True)
class Workload:
    name: str
    hidden: int
    n_experts: int
    top_k: int
    inter: int
    shared_inter: int
    dtype: int
    has_shared_gate: int
    x_std: float
    w_std: float
    router_std: float
    T: int = 1
    layers: int = 1
    routing: str = "normal"          # "normal" | "zipf"
    zipf_s: float = 1.1
    norm_topk: int = 1
    preset_id: int = 0
    t_values: tuple = field(default=())

    @property
    def torch_dtype(self):
        return _TORCH_DT[self.dtype]

    def layer_bytes(self) -> int:
        """Bytes of one layer's weights as stored in HBM."""
        H, E, I, Is = self.hidden, self.n_experts, self.inter, self.shared_inter
        n = E * H + E * 2 * I * H + E * H * I + 2 * Is * H + H * Is + (H if self.has_shared_gate else 0)
        return 2 * n


PRESETS = {
    "tiny": Workload("tiny", 256, 16, 2, 64, 0, F16, 0, 0.02, 0.02, 0.1,
                     T=1, layers=1, preset_id=1),
    "sharded_decode": Workload("sharded_decode", 2048, 256, 8, 128, 128, F16, 0, 1.0, 0.02, 0.02,
                               T=1, layers=36, preset_id=2),
    "full_decode": Workload("full_decode", 2048, 256, 8, 512, 512, BF16, 1, 1.0, 0.02, 0.02,
                            T=1, layers=36, preset_id=3),
    "small_batch": Workload("small_batch", 2048, 256, 8, 512, 512, BF16, 1, 1.0, 0.02, 0.02,
                            T=16, layers=36, routing="zipf", preset_id=4, t_values=(2, 4, 8, 16, 64)),
    "chunked_prefill": Workload("chunked_prefill", 2048, 256, 8, 512, 512, BF16, 1, 1.0, 0.02,
                                1.0 / math.sqrt(2048), T=512, layers=4, preset_id=5,
                                t_values=(512, 4096)),
}


def workload(name: str, **over) -> Workload:
    return replace(PRESETS[name], **over)


def seed_of(wl: Workload, layer: int, tensor_id: int, base: int = 0) -> int:
    return base + 1000 * wl.preset_id + 16 * layer + tensor_id


# tensor ids inside one layer
_X, _WR, _W13, _W2, _SW13, _SW2, _SWG, _PERM = range(8)


def _normal(shape, std, seed, device, dtype):
    """N(0, std^2) drawn in fp32 from a seeded generator, rounded to ``dtype``."""
    if torch.device(device).type == "cuda":
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        out = torch.empty(shape, dtype=dtype, device=device)
        flat = out.view(-1)
        chunk = 1 << 27
        for s in range(0, flat.numel(), chunk):
            n = min(chunk, flat.numel() - s)
            flat[s:s + n] = (torch.randn(n, generator=g, device=device, dtype=torch.float32) * std).to(dtype)
        return out
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal(size=int(np.prod(shape)), dtype=np.float32) * np.float32(std)
    return torch.from_numpy(a).reshape(shape).to(dtype)


def zipf_ranks(wl: Workload, layer: int, base: int = 0) -> np.ndarray:
    """Seeded permutation rank (1..E) of every expert for the Zipf workload."""
    rng = np.random.Generator(np.random.PCG64(seed_of(wl, layer, _PERM, base)))
    return rng.permutation(wl.n_experts) + 1


def make_layer(wl: Workload, layer: int = 0, T: int | None = None, device="cpu",
               seed_base: int = 0, x_only: bool = False, weights_only: bool = False) -> dict:
    """One layer's seeded inputs as torch tensors on ``device``."""
    T = wl.T if T is None else T
    H, E, I, Is = wl.hidden, wl.n_experts, wl.inter, wl.shared_inter
    dt = wl.torch_dtype
    d = {}
    if not weights_only:
        x = _normal((T, H), wl.x_std, seed_of(wl, layer, _X, seed_base), device, dt)
        if wl.routing == "zipf":
            x[:, 0] = 1.0
        d["x"] = x
    if x_only:
        return d
    d["router_w"] = make_router(wl, layer, device, seed_base)
    d["w13"] = _normal((E, 2 * I, H), wl.w_std, seed_of(wl, layer, _W13, seed_base), device, dt)
    d["w2"] = _normal((E, H, I), wl.w_std, seed_of(wl, layer, _W2, seed_base), device, dt)
    if Is > 0:
        d["shared_w13"] = _normal((2 * Is, H), wl.w_std, seed_of(wl, layer, _SW13, seed_base), device, dt)
        d["shared_w2"] = _normal((H, Is), wl.w_std, seed_of(wl, layer, _SW2, seed_base), device, dt)
    else:
        d["shared_w13"] = None
        d["shared_w2"] = None
    if wl.has_shared_gate:
        d["shared_gate_w"] = _normal((H,), wl.w_std, seed_of(wl, layer, _SWG, seed_base), device, dt)
    else:
        d["shared_gate_w"] = None
    return d


def make_router(wl: Workload, layer: int, device, seed_base: int = 0):
    """One layer's router weights [E, H] (with the Zipf column for ``zipf``)."""
    wr = _normal((wl.n_experts, wl.hidden), wl.router_std, seed_of(wl, layer, _WR, seed_base), device,
                 wl.torch_dtype)
    if wl.routing == "zipf":
        r = torch.from_numpy(zipf_ranks(wl, layer, seed_base).astype(np.float64))
        wr[:, 0] = (-wl.zipf_s * torch.log(r)).to(wl.torch_dtype).to(wr.device)
    return wr


def make_x(wl: Workload, layer: int, T: int, device, seed_base: int = 0):
    return make_layer(wl, layer, T, device, seed_base, x_only=True)["x"]


def bits(t) -> np.ndarray | None:
    """Raw uint16 bit patterns of a 2-byte float tensor (copied to host)."""
    if t is None:
        return None
    if t.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("bits() wants an fp16/bf16 tensor")
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(b: np.ndarray, dtype: int, device="cpu"):
    """Tensor of storage dtype ``dtype`` holding the given uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(_TORCH_DT[dtype])
    return t.to(device)
