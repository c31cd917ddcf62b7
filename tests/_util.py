"""Shared helpers of the GPU parity tests: oracle calls on the same bytes and
the tolerance the block is judged by."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import moe_synth
import oracle

# Tolerance for fp32 accumulation over fp16/bf16 weights, checked against the
# fp64 oracle: max |err| <= 1e-2 * max |ref| and sum |err| / sum |ref| <= 2e-3.
MAX_ERR_FRAC = 1e-2
REL_L1 = 2e-3


def ocfg(wl):
    return oracle.OracleCfg(wl.hidden, wl.n_experts, wl.top_k, wl.inter, wl.shared_inter, wl.dtype,
                            wl.norm_topk, wl.has_shared_gate)


def oracle_full(wl, d):
    """Oracle on a whole layer whose tensors are on the host (small cases)."""
    b = moe_synth.bits
    return oracle.moe_forward(ocfg(wl), b(d["x"]), b(d["router_w"]), b(d["w13"]), b(d["w2"]),
                              b(d["shared_w13"]), b(d["shared_w2"]), b(d["shared_gate_w"]))


def oracle_sampled(wl, d, tokens):
    """Oracle for selected tokens of a layer whose tensors are on the GPU: the
    oracle first routes each token, then only the experts it selects are
    copied to the host."""
    b = moe_synth.bits
    c = ocfg(wl)
    x = b(d["x"])
    wr = b(d["router_w"])
    res = {"ids": [], "w": [], "logits": [], "out": []}
    for t in tokens:
        lg, ids, _ = oracle.router(c, x[t], wr)
        w13 = {int(e): b(d["w13"][int(e)]) for e in ids}
        w2 = {int(e): b(d["w2"][int(e)]) for e in ids}
        r = oracle.moe_forward(c, x[t:t + 1], wr, w13, w2, b(d["shared_w13"]), b(d["shared_w2"]),
                               b(d["shared_gate_w"]))
        for key in res:
            res[key].append(r[key][0])
    return {key: np.stack(v) for key, v in res.items()}


def oracle_tokens(wl, d, tokens):
    """Oracle for the listed tokens of a layer whose tensors are on the GPU.
    The layer is copied to the host once; the tokens are split over a thread
    pool (each oracle call runs in C with the GIL released).  Rows of the
    result follow the order of ``tokens``."""
    b = moe_synth.bits
    c = ocfg(wl)
    x = b(d["x"])
    args = [b(d[k]) for k in ("router_w", "w13", "w2", "shared_w13", "shared_w2", "shared_gate_w")]
    tokens = [int(t) for t in tokens]
    n = max(1, min(64, os.cpu_count() or 1))
    step = max(1, -(-len(tokens) // (4 * n)))
    chunks = [tokens[i:i + step] for i in range(0, len(tokens), step)]

    def run(ch):
        return oracle.moe_forward(c, np.ascontiguousarray(x[ch]), *args)

    with ThreadPoolExecutor(n) as ex:
        parts = list(ex.map(run, chunks))
    return {key: np.concatenate([p[key] for p in parts]) for key in ("ids", "w", "logits", "out")}


def check_tokens(ids, w, out, ref, tokens, k, min_exact=0.8):
    """GPU rows ``tokens`` against oracle rows 0.. (same order): ids
    bit-exact and weights to 1e-4 wherever the oracle's adjacent-rank gaps
    exceed 1e-4 (at least ``min_exact`` of the tokens must qualify), every
    token's output within the tolerance, and the whole set too."""
    ids_g = ids[tokens].cpu().numpy()
    w_g = w[tokens].cpu().numpy()
    gaps = min_rank_gap(ref["logits"], k)
    sure = gaps > 1e-4
    assert np.array_equal(ids_g[sure], ref["ids"][sure]), np.nonzero((ids_g != ref["ids"]).any(-1) & sure)
    np.testing.assert_allclose(w_g[sure], ref["w"][sure], rtol=1e-4, atol=1e-6)
    assert sure.sum() >= max(1, int(min_exact * len(tokens))), (sure.sum(), len(tokens))
    o = out[tokens].detach().float().cpu().double().numpy()
    for i in range(len(tokens)):
        parity(o[i], ref["out"][i])
    return parity(o, ref["out"])


def parity(got, ref, max_err_frac=MAX_ERR_FRAC, rel_l1=REL_L1):
    """Assert the tolerance; returns (max_err / max_ref, rel_l1)."""
    g = got.detach().float().cpu().double().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), "non-finite output"
    err = np.abs(g - r)
    frac = err.max() / max(np.abs(r).max(), 1e-300)
    rel = err.sum() / max(np.abs(r).sum(), 1e-300)
    assert frac <= max_err_frac, f"max|err|/max|ref| = {frac:.3e} > {max_err_frac}"
    assert rel <= rel_l1, f"relative L1 = {rel:.3e} > {rel_l1}"
    return frac, rel


def min_rank_gap(logits, k):
    """Smallest gap between adjacent ranks 0..k (fp64 logits), per token."""
    s = -np.sort(-np.asarray(logits, np.float64), axis=-1)[..., : k + 1]
    return np.min(s[..., :-1] - s[..., 1:], axis=-1)


def fp32_topk(logits32, k):
    """Top-k of fp32 logits by (value desc, index asc), numpy's stable sort."""
    l = np.asarray(logits32, np.float32)
    order = np.argsort(-l, axis=-1, kind="stable")
    return order[..., :k].astype(np.int32)


def _check_one_token(ids, w, out, ref, k, t=0, i=0):
    """Token t of a GPU result against row i of an oracle result: ids bit-exact
    where the oracle's adjacent-rank gaps exceed 1e-4, weights to 1e-4
    relative, output within the tolerance."""
    if min_rank_gap(ref["logits"][i], k) > 1e-4:
        assert np.array_equal(ids[t].cpu().numpy(), ref["ids"][i]), (ids[t], ref["ids"][i])
        np.testing.assert_allclose(w[t].cpu().numpy(), ref["w"][i], rtol=1e-4, atol=1e-6)
    parity(out[t:t + 1], ref["out"][i:i + 1])
