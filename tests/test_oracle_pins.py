"""Pins of the oracle against facts that do not come from the oracle itself.

Each test ties one oracle function to something the pages or the mathematics
fix: exhaustive decoding against numpy/torch conversions, the pages' known-data
value, closed forms of the SiLU-gated FFN, brute-force enumeration of routing,
exact special cases (zero input, duplicated router rows, zero gate), exact
linearity, and the pages' second (copy-out) formulation.  A plausible slip in
the oracle (swapped gate/up rows, a transposed W2, a dropped shared term, a
wrong tie-break, a softmax over the wrong set) fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax as sp_softmax

import oracle
from oracle import OracleCfg, F16, BF16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            vals[k] = float(v)
    return vals


def _bits_of(values, dtype):
    t = torch.as_tensor(np.asarray(values, np.float32))
    t = t.to(torch.float16 if dtype == F16 else torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _to64(bits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    t = t.view(torch.float16 if dtype == F16 else torch.bfloat16)
    return t.to(torch.float64).numpy()


def _rand_case(rng, H, E, k, I, Is, dtype, gate, T, std=0.3):
    def r(*shape):
        return _bits_of(rng.standard_normal(shape) * std, dtype)
    d = dict(x=r(T, H), wr=r(E, H), w13=r(E, 2 * I, H), w2=r(E, H, I))
    d["sw13"] = r(2 * Is, H) if Is else None
    d["sw2"] = r(H, Is) if Is else None
    d["swg"] = r(H) if gate else None
    return d


# --------------------------------------------------------------- decoding
def test_decode_f16_exhaustive():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle.decode(int(b), F16) for b in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_decode_bf16_exhaustive():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.decode(int(b), BF16) for b in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# --------------------------------------------------- the pages' known data
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_known_data_w2_gives_128(dtype):
    g = _read_golden("known_data_w2.txt")
    I, H, k = int(g["inter"]), int(g["hidden"]), int(g["top_k"])
    E = 16
    cfg = OracleCfg(hidden=H, n_experts=E, top_k=k, inter=I, dtype=dtype)
    w2 = np.broadcast_to(_bits_of([g["w2_value"]], dtype)[0], (E, H, I)).copy()
    act = np.full((k, I), g["act_value"])
    ids = np.arange(k, dtype=np.int32)[::-1].copy()
    w = np.array([0.5, 0.25, 0.125, 0.0625, 0.03125, 0.015625, 0.0078125, 0.0078125])
    assert w.sum() == 1.0
    out = oracle.w2_combine(cfg, act, ids, w, w2)
    assert np.all(out == g["expected_per_output"])
    assert not np.any(out == g["wrong_value_reported"])


# ------------------------------------- W2 layout [E, H, I] on random activations
def _rank1_w2(E, H, I, dtype, rng):
    """W2[e, h, i] = s_e * a_h * b_i with small dyadic factors, exact in fp16
    and bf16 (each product has at most 7 significant bits)."""
    a = 1 + rng.integers(0, 4, H) / 4
    b = 1 + rng.integers(0, 8, I) / 8
    s = 2.0 ** rng.integers(-2, 3, E)
    w = s[:, None, None] * a[None, :, None] * b[None, None, :]
    bits = _bits_of(w, dtype)
    assert np.array_equal(_to64(bits, dtype), w)
    return bits, a, b, s


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_w2_combine_rank_one_w2_on_random_activations(dtype):
    """The down projection reads row h of expert e as the I contiguous values
    W2[e, h, 0:I] (work log Parts 4 and 10: W2[expert_ids[k], h, :]).  With
    a rank-one W2 = s_e a_h b_i the routed output is a_h times one scalar,
    sum_j w_j s_{id_j} sum_i b_i act[j, i], for any activation.  A transposed
    or shifted index (H != I here) breaks the proportionality."""
    rng = np.random.default_rng(11)
    H, I, E, k = 40, 24, 6, 3
    cfg = OracleCfg(hidden=H, n_experts=E, top_k=k, inter=I, dtype=dtype)
    w2, a, b, s = _rank1_w2(E, H, I, dtype, rng)
    act = rng.standard_normal((k, I))
    ids = rng.permutation(E)[:k].astype(np.int32)
    w = rng.random(k) + 0.1
    out = oracle.w2_combine(cfg, act, ids, w, w2)
    scalar = sum(w[j] * s[ids[j]] * float(np.dot(b, act[j])) for j in range(k))
    np.testing.assert_allclose(out, a * scalar, rtol=1e-12, atol=0)


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("Is,gate", [(0, 0), (16, 1)])
def test_forward_rank_one_w2_output_is_proportional(dtype, Is, gate):
    """Whole block on random x, router and W13 with rank-one down projections
    (routed W2[e, h, i] = s_e a_h b_i, shared Ws2[h, i] = a_h c_i): every
    token's output is a_h times a per-token scalar, whatever the routing and
    the activations.  Pins the [E, H, I] and [H, Is] layouts of the forward
    pass on random data (the closed-form tests use W2 = 1, which any index
    order satisfies)."""
    rng = np.random.default_rng(12)
    H, E, k, I, T = 40, 8, 3, 24, 3
    d = _rand_case(rng, H, E, k, I, Is, dtype, gate, T)
    d["w2"], a, b, s = _rank1_w2(E, H, I, dtype, rng)
    if Is:
        c = 1 + rng.integers(0, 8, Is) / 8
        d["sw2"] = _bits_of(a[:, None] * c[None, :], dtype)
    cfg = OracleCfg(hidden=H, n_experts=E, top_k=k, inter=I, shared_inter=Is, dtype=dtype,
                    has_shared_gate=gate)
    r = oracle.moe_forward(cfg, d["x"], d["wr"], d["w13"], d["w2"], d["sw13"], d["sw2"], d["swg"])
    ratio = r["out"] / a[None, :]
    assert np.all(np.abs(ratio[:, 0]) > 1e-6)
    np.testing.assert_allclose(ratio, np.repeat(ratio[:, :1], H, axis=1), rtol=1e-12, atol=0)


# ----------------------------------------------------------- closed forms
def _closed_form_case(H, E, k, I, Is, c, cs, dtype, gate, rng, T=2):
    """x = 1; gate rows = c/H, up rows = 1/H; W2 = 1 -> every routed expert
    yields y_h = I * silu(c) whatever the routing; shared expert likewise with cs."""
    one = _bits_of([1.0], dtype)[0]
    x = np.full((T, H), one, np.uint16)
    wr = _bits_of(rng.standard_normal((E, H)) * 0.1, dtype)
    w13 = np.empty((E, 2 * I, H), np.uint16)
    w13[:, :I, :] = _bits_of([c / H], dtype)[0]
    w13[:, I:, :] = _bits_of([1.0 / H], dtype)[0]
    w2 = np.full((E, H, I), one, np.uint16)
    d = dict(x=x, wr=wr, w13=w13, w2=w2, sw13=None, sw2=None, swg=None)
    if Is:
        sw13 = np.empty((2 * Is, H), np.uint16)
        sw13[:Is] = _bits_of([cs / H], dtype)[0]
        sw13[Is:] = _bits_of([1.0 / H], dtype)[0]
        d["sw13"] = sw13
        d["sw2"] = np.full((H, Is), one, np.uint16)
        if gate:
            d["swg"] = np.zeros(H, np.uint16)          # sigmoid(0) = 1/2 exactly
    return d


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("shared,gate", [(0, 0), (64, 0), (64, 1)])
def test_closed_form_silu_ffn(dtype, shared, gate):
    rng = np.random.default_rng(7)
    H, E, k, I, c, cs = 256, 16, 4, 32, 4.0, 2.0
    cfg = OracleCfg(H, E, k, I, shared, dtype, 1, gate)
    d = _closed_form_case(H, E, k, I, shared, c, cs, dtype, gate, rng)
    res = oracle.moe_forward(cfg, d["x"], d["wr"], d["w13"], d["w2"], d["sw13"], d["sw2"], d["swg"])
    silu = lambda v: v / (1.0 + math.exp(-v))
    expect = I * silu(c)
    if shared:
        expect += (0.5 if gate else 1.0) * shared * silu(cs)
    np.testing.assert_allclose(res["out"], expect, rtol=1e-13, atol=0)


def test_closed_form_sigmoid_gate_saturates():
    """wg = 1/16 with x = 1, H = 256 gives x.wg = 16: g = 1/(1+e^-16)."""
    rng = np.random.default_rng(3)
    H, E, k, I, Is = 256, 8, 2, 16, 16
    cfg = OracleCfg(H, E, k, I, Is, F16, 1, 1)
    d = _closed_form_case(H, E, k, I, Is, 1.0, 3.0, F16, 1, rng)
    d["swg"] = np.full(H, _bits_of([1.0 / 16], F16)[0], np.uint16)
    res = oracle.moe_forward(cfg, d["x"], d["wr"], d["w13"], d["w2"], d["sw13"], d["sw2"], d["swg"])
    silu = lambda v: v / (1.0 + math.exp(-v))
    expect = I * silu(1.0) + Is * silu(3.0) / (1.0 + math.exp(-16.0))
    np.testing.assert_allclose(res["out"], expect, rtol=1e-13)


def test_gate_and_up_rows_are_not_interchangeable():
    """Swapping the halves of W13 changes silu(c)*1 into silu(1)*c: the closed
    form above would catch an oracle that read gate/up the other way round."""
    rng = np.random.default_rng(5)
    H, E, k, I = 256, 8, 2, 16
    cfg = OracleCfg(H, E, k, I, 0, F16)
    d = _closed_form_case(H, E, k, I, 0, 4.0, 0.0, F16, 0, rng, T=1)
    w13s = d["w13"].copy()
    w13s[:, :I], w13s[:, I:] = d["w13"][:, I:], d["w13"][:, :I]
    a = oracle.moe_forward(cfg, d["x"], d["wr"], d["w13"], d["w2"])["out"]
    b = oracle.moe_forward(cfg, d["x"], d["wr"], w13s, d["w2"])["out"]
    silu = lambda v: v / (1.0 + math.exp(-v))
    np.testing.assert_allclose(a, I * silu(4.0), rtol=1e-13)
    np.testing.assert_allclose(b, I * 4.0 * silu(1.0), rtol=1e-13)


# --------------------------------------------------------------- routing
def _brute_force_topk(logits, k):
    E = len(logits)
    best, best_key = None, None
    for tup in itertools.permutations(range(E), k):
        key = [v for e in tup for v in (logits[e], -e)]
        if best_key is None or key > best_key:
            best, best_key = tup, key
    return list(best)


@pytest.mark.parametrize("E,k", [(8, 3), (16, 2), (6, 6)])
def test_routing_brute_force_with_ties(E, k):
    """Logits on a coarse dyadic grid (exact in fp16 and in double) so ties are
    frequent; the oracle's ids must equal the brute-force optimum over all
    ordered k-tuples under (logit desc, index asc)."""
    H = 16
    rng = np.random.default_rng(11 + E + k)
    one = _bits_of([1.0], F16)[0]
    x = np.full(H, one, np.uint16)
    for trial in range(40):
        q = rng.integers(-2, 3, size=(E, H)) / 8.0        # sums are multiples of 1/8
        wr = _bits_of(q, F16)
        exact = q.sum(axis=1)
        cfg = OracleCfg(H, E, k, 8, 0, F16, norm_topk=1)
        lg, ids, w = oracle.router(cfg, x, wr)
        assert np.array_equal(lg, exact)
        assert list(ids) == _brute_force_topk(list(exact), k)
        np.testing.assert_allclose(w, sp_softmax(exact[ids]), rtol=1e-14)
        assert abs(w.sum() - 1.0) < 1e-15
        assert np.all(np.diff(w) <= 0)


def test_routing_zero_input_all_tie():
    """x = 0 makes every logit 0: ids are 0..k-1 and every weight is 1/k."""
    E, k, H = 16, 4, 64
    rng = np.random.default_rng(1)
    wr = _bits_of(rng.standard_normal((E, H)), F16)
    x = np.zeros(H, np.uint16)
    lg, ids, w = oracle.router(OracleCfg(H, E, k, 8, 0, F16), x, wr)
    assert np.all(lg == 0)
    assert list(ids) == list(range(k))
    assert np.all(w == 1.0 / k)


def test_routing_duplicated_rows_lower_index_first():
    """Experts 2, 7 and 9 share one router row bit for bit and that row is
    aligned with x, so they hold the three largest (equal) logits: the ranks
    must come out as 2, 7, 9 (lower index first)."""
    E, k, H = 12, 5, 32
    rng = np.random.default_rng(2)
    xf = rng.standard_normal(H)
    x = _bits_of(xf, BF16)
    base = _bits_of(rng.standard_normal((E, H)) * 0.05, BF16)
    top = _bits_of(xf * 0.5, BF16)
    for e in (9, 2, 7):
        base[e] = top
    lg, ids, w = oracle.router(OracleCfg(H, E, k, 8, 0, BF16), x, base)
    assert lg[2] == lg[7] == lg[9]
    assert list(ids[:3]) == [2, 7, 9]
    assert w[0] == w[1] == w[2]
    assert list(ids) == _brute_force_topk(list(lg), k)


def test_softmax_over_all_experts_without_renorm():
    """With norm_topk = 0 and k = E every expert is selected and the weights
    are the plain softmax of the logits (scipy's routine, logits by numpy)."""
    H, E = 64, 10
    rng = np.random.default_rng(4)
    x = _bits_of(rng.standard_normal(H), F16)
    wr = _bits_of(rng.standard_normal((E, H)) * 0.2, F16)
    cfg = OracleCfg(H, E, E, 8, 0, F16, norm_topk=0)
    lg, ids, w = oracle.router(cfg, x, wr)
    ref_lg = _to64(wr, F16) @ _to64(x, F16)
    np.testing.assert_allclose(lg, ref_lg, rtol=1e-13, atol=1e-13)
    p = sp_softmax(ref_lg)
    np.testing.assert_allclose(w, p[ids], rtol=1e-12)
    assert abs(w.sum() - 1.0) < 1e-13
    # top-3 without renormalisation keeps the full-softmax values
    cfg3 = OracleCfg(H, E, 3, 8, 0, F16, norm_topk=0)
    _, ids3, w3 = oracle.router(cfg3, x, wr)
    np.testing.assert_allclose(w3, p[ids3], rtol=1e-12)
    assert w3.sum() < 1.0


# ------------------------------------------ formulations, structure, linearity
@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("Is,gate", [(0, 0), (24, 0), (24, 1)])
def test_direct_equals_copy_out_formulation(dtype, Is, gate):
    """The direct-routed formulation equals the pages' fallback (index_select,
    dense linear, SiluAndMul, bmm, weighted sum)."""
    rng = np.random.default_rng(100 + dtype + Is + gate)
    H, E, k, I, T = 64, 12, 3, 16, 3
    cfg = OracleCfg(H, E, k, I, Is, dtype, 1, gate)
    d = _rand_case(rng, H, E, k, I, Is, dtype, gate, T)
    a = oracle.moe_forward(cfg, d["x"], d["wr"], d["w13"], d["w2"], d["sw13"], d["sw2"], d["swg"])["out"]
    b = oracle.moe_forward_gather(cfg, d["x"], d["wr"], d["w13"], d["w2"], d["sw13"], d["sw2"], d["swg"])
    scale = np.abs(a).max()
    assert np.abs(a - b).max() <= 1e-12 * scale


def test_independent_numpy_formulation():
    """A third formulation with numpy library primitives (matmul, exp) on the
    same bytes; catches transposed operands and dropped terms."""
    rng = np.random.default_rng(9)
    H, E, k, I, Is, T = 48, 10, 3, 8, 16, 4
    cfg = OracleCfg(H, E, k, I, Is, BF16, 1, 1)
    d = _rand_case(rng, H, E, k, I, Is, BF16, 1, T)
    res = oracle.moe_forward(cfg, d["x"], d["wr"], d["w13"], d["w2"], d["sw13"], d["sw2"], d["swg"])
    X = _to64(d["x"], BF16)
    Wr, W13, W2 = _to64(d["wr"], BF16), _to64(d["w13"], BF16), _to64(d["w2"], BF16)
    S13, S2, G = _to64(d["sw13"], BF16), _to64(d["sw2"], BF16), _to64(d["swg"], BF16)
    silu = lambda v: v / (1.0 + np.exp(-v))
    for t in range(T):
        lg = Wr @ X[t]
        ids = res["ids"][t]
        np.testing.assert_allclose(res["logits"][t], lg, rtol=1e-12, atol=1e-12)
        w = sp_softmax(lg[ids])
        out = np.zeros(H)
        for j, e in enumerate(ids):
            gu = W13[e] @ X[t]
            out += w[j] * (W2[e] @ (silu(gu[:I]) * gu[I:]))
        sgu = S13 @ X[t]
        out += (1.0 / (1.0 + np.exp(-(G @ X[t])))) * (S2 @ (silu(sgu[:Is]) * sgu[Is:]))
        np.testing.assert_allclose(res["out"][t], out, rtol=1e-10, atol=1e-12)


def test_scaling_w2_by_two_doubles_output_exactly():
    rng = np.random.default_rng(12)
    H, E, k, I = 64, 8, 2, 16
    cfg = OracleCfg(H, E, k, I, 0, F16)
    d = _rand_case(rng, H, E, k, I, 0, F16, 0, 2)
    w2x2 = _bits_of(_to64(d["w2"], F16) * 2.0, F16)
    a = oracle.moe_forward(cfg, d["x"], d["wr"], d["w13"], d["w2"])["out"]
    b = oracle.moe_forward(cfg, d["x"], d["wr"], d["w13"], w2x2)["out"]
    assert np.array_equal(b, 2.0 * a)


def test_zero_routed_w2_leaves_shared_only():
    rng = np.random.default_rng(13)
    H, E, k, I, Is = 256, 8, 2, 16, 32
    cfg = OracleCfg(H, E, k, I, Is, BF16, 1, 0)
    d = _closed_form_case(H, E, k, I, Is, 4.0, 2.0, BF16, 0, rng, T=1)
    d["w2"] = np.zeros_like(d["w2"])
    res = oracle.moe_forward(cfg, d["x"], d["wr"], d["w13"], d["w2"], d["sw13"], d["sw2"])
    np.testing.assert_allclose(res["out"], Is * 2.0 / (1.0 + math.exp(-2.0)), rtol=1e-13)


def test_zero_gate_vector_halves_shared_exactly():
    rng = np.random.default_rng(14)
    H, E, k, I, Is = 64, 8, 2, 16, 16
    d = _rand_case(rng, H, E, k, I, Is, F16, 0, 2)
    d["w2"] = np.zeros_like(d["w2"])
    plain = oracle.moe_forward(OracleCfg(H, E, k, I, Is, F16, 1, 0), d["x"], d["wr"], d["w13"], d["w2"],
                               d["sw13"], d["sw2"])["out"]
    gated = oracle.moe_forward(OracleCfg(H, E, k, I, Is, F16, 1, 1), d["x"], d["wr"], d["w13"], d["w2"],
                               d["sw13"], d["sw2"], np.zeros(H, np.uint16))["out"]
    assert np.array_equal(gated, 0.5 * plain)


def test_tokens_are_independent_and_permute():
    rng = np.random.default_rng(15)
    H, E, k, I, Is, T = 64, 8, 3, 16, 16, 5
    cfg = OracleCfg(H, E, k, I, Is, F16, 1, 1)
    d = _rand_case(rng, H, E, k, I, Is, F16, 1, T)
    full = oracle.moe_forward(cfg, d["x"], d["wr"], d["w13"], d["w2"], d["sw13"], d["sw2"], d["swg"])
    perm = rng.permutation(T)
    pr = oracle.moe_forward(cfg, d["x"][perm], d["wr"], d["w13"], d["w2"], d["sw13"], d["sw2"], d["swg"])
    assert np.array_equal(pr["out"], full["out"][perm])
    assert np.array_equal(pr["ids"], full["ids"][perm])
    for t in range(T):
        one = oracle.moe_forward(cfg, d["x"][t:t + 1], d["wr"], d["w13"], d["w2"], d["sw13"], d["sw2"], d["swg"])
        assert np.array_equal(one["out"][0], full["out"][t])


def test_missing_selected_expert_is_an_error():
    rng = np.random.default_rng(16)
    H, E, k, I = 32, 6, 2, 8
    cfg = OracleCfg(H, E, k, I, 0, F16)
    d = _rand_case(rng, H, E, k, I, 0, F16, 0, 1)
    _, ids, _ = oracle.router(cfg, d["x"][0], d["wr"])
    w13 = {e: d["w13"][e] for e in range(E) if e != ids[1]}
    w2 = {e: d["w2"][e] for e in range(E)}
    with pytest.raises(RuntimeError):
        oracle.moe_forward(cfg, d["x"], d["wr"], w13, w2)
    w13[int(ids[1])] = d["w13"][ids[1]]
    a = oracle.moe_forward(cfg, d["x"], d["wr"], w13, w2)["out"]
    b = oracle.moe_forward(cfg, d["x"], d["wr"], d["w13"], d["w2"])["out"]
    assert np.array_equal(a, b)


def test_pages_shard_traffic_matches_layout():
    """The pages' 8.4 MB / 4.2 MB per-layer traffic is exactly the selected
    rows of the stacked layout the oracle indexes (k experts x 2I rows x H,
    and k x H rows x I, 2-byte elements)."""
    g = _read_golden("sharded_roofline_bytes.txt")
    H, k, I = 2048, 8, 128
    w13 = k * 2 * I * H * 2
    w2 = k * H * I * 2
    assert round(w13 / 1e6, 1) == g["w13_selected_mb"]
    assert round(w2 / 1e6, 1) == g["w2_selected_mb"]
    assert round((w13 + w2) / 1e6, 1) == g["total_mb"]
    flops = 2 * (w13 + w2) / 2
    assert round(flops / (w13 + w2), 1) == g["flop_per_byte"]
