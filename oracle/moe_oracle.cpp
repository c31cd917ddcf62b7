// moe_oracle.cpp — reference oracle for the decode-step MoE block.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
// call this file: only the tests, the package's smoke check and the CPU
// baseline leg of the benchmark do.  It shares no code, header, table or
// constant with the CUDA library; its only common input with the GPU path is
// the raw fp16/bf16 bytes of the seeded synthetic tensors.
//
// Plain, slow, obviously correct: single-threaded C++17, every sum in
// IEEE double, loops in the order the method states them, libm exp().
//
// Sources (the pages this restates; no listing is copied):
//  * "BI-V100 inference work log" (kernel_worklog), Part 3 — the PyTorch
//    fallback MoE path: gate, topk, softmax, index_select of the selected
//    experts' W13/W2, F.linear, SiluAndMul, bmm over the k experts, weighted
//    sum; plus the shared expert (gate_up + SiluAndMul + down).
//  * same page, Part 4 and Part 10 — the "direct_routed" formulation that
//    indexes W13[expert_ids[k], row, :] and W2[expert_ids[k], h, :] in place
//    instead of copying; shapes x(1,H), gate_up(k,2I), W2 rows of I.
//  * same page, Part 1 — the known-data W2 check (all-ones activation, unit
//    weights, a 128-long dot product gives 128.0).
//  * "Decode throughput analysis report" (decode_analysis_report), code-level
//    profiling section — T>1 tokens are independent rows; the tiny-batch path
//    flattens T*k (token, expert) pairs.
// Readings where the pages are silent (each listed in the design notes):
//  gate rows are W13[e, 0:I), up rows W13[e, I:2I), act = silu(gate)*up;
//  softmax over all E logits, top-k by (logit desc, index asc), then the k
//  weights renormalised to sum 1 when norm_topk is set; the shared expert's
//  output is scaled by sigmoid(x . wg) when a gate vector is given, else 1.
//
// Parity status: every function here is pinned by tests/test_oracle_pins.py
// (exhaustive decode checks, closed forms, brute-force routing, the pages'
// known-data value, and a second independent formulation).  The exact
// rounding of the fp64 sums is not pinned beyond those cases.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <algorithm>

namespace {

// dtype codes accepted by this oracle (its own numbering).
constexpr int32_t ORC_F16 = 1;
constexpr int32_t ORC_BF16 = 2;

// IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits.
double decode_f16(uint16_t b) {
  const int s = b >> 15;
  const int e = (b >> 10) & 0x1f;
  const int m = b & 0x3ff;
  double v;
  if (e == 0) {
    v = std::ldexp(static_cast<double>(m), -24);          // subnormal: m * 2^-24
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = std::ldexp(static_cast<double>(m + 1024), e - 25); // (1 + m/1024) * 2^(e-15)
  }
  return s ? -v : v;
}

// bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits (the top half of binary32).
double decode_bf16(uint16_t b) {
  const int s = b >> 15;
  const int e = (b >> 7) & 0xff;
  const int m = b & 0x7f;
  double v;
  if (e == 0) {
    v = std::ldexp(static_cast<double>(m), -133);           // subnormal: m/128 * 2^-126
  } else if (e == 255) {
    v = m ? NAN : INFINITY;
  } else {
    v = std::ldexp(static_cast<double>(m + 128), e - 134);  // (1 + m/128) * 2^(e-127)
  }
  return s ? -v : v;
}

double decode(uint16_t b, int32_t dtype) {
  return dtype == ORC_BF16 ? decode_bf16(b) : decode_f16(b);
}

double silu(double v) { return v / (1.0 + std::exp(-v)); }
double sigmoid(double v) { return 1.0 / (1.0 + std::exp(-v)); }

}  // namespace

extern "C" {

// The oracle's own description of one MoE block.
struct oracle_cfg {
  int32_t hidden;           // H
  int32_t n_experts;        // E
  int32_t top_k;            // k
  int32_t inter;            // I, per routed expert
  int32_t shared_inter;     // Is, 0 = no shared expert
  int32_t dtype;            // 1 = fp16, 2 = bf16 (bytes of every input tensor)
  int32_t norm_topk;        // 1 = renormalise the k routing weights to sum 1
  int32_t has_shared_gate;  // 1 = shared output scaled by sigmoid(x . wg)
};

// Status codes.
enum { ORC_OK = 0, ORC_BAD_ARG = 1, ORC_MISSING_EXPERT = 2 };

double oracle_decode(uint16_t bits, int32_t dtype) { return decode(bits, dtype); }

int32_t oracle_version(void) { return 1; }

static bool cfg_ok(const oracle_cfg* c) {
  return c && c->hidden > 0 && c->n_experts > 0 && c->top_k > 0 &&
         c->top_k <= c->n_experts && c->inter > 0 && c->shared_inter >= 0 &&
         (c->dtype == ORC_F16 || c->dtype == ORC_BF16);
}

// Router for one token ("gate", then "topk" and "softmax" in the fallback
// path of the work log's Part 3).
//   logits[e] = sum_h x[h] * wr[e, h]
//   ids       = the k experts ranked by (logit desc, index asc)
//   w[j]      = softmax(logits)[ids[j]], renormalised over the k when norm_topk
int oracle_router_token(const oracle_cfg* c, const uint16_t* x, const uint16_t* wr,
                        double* logits, int32_t* ids, double* w) {
  if (!cfg_ok(c) || !x || !wr || !logits || !ids || !w) return ORC_BAD_ARG;
  const int H = c->hidden, E = c->n_experts, k = c->top_k;
  for (int e = 0; e < E; ++e) {
    double acc = 0.0;
    for (int h = 0; h < H; ++h)
      acc += decode(x[h], c->dtype) * decode(wr[static_cast<size_t>(e) * H + h], c->dtype);
    logits[e] = acc;
  }
  // Rank: a stable sort on "logit greater" keeps equal logits in index order.
  std::vector<int32_t> order(E);
  for (int e = 0; e < E; ++e) order[e] = e;
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t a, int32_t b) { return logits[a] > logits[b]; });
  double mx = logits[order[0]];
  double z = 0.0;
  for (int e = 0; e < E; ++e) z += std::exp(logits[e] - mx);
  double wsum = 0.0;
  for (int j = 0; j < k; ++j) {
    ids[j] = order[j];
    w[j] = std::exp(logits[order[j]] - mx) / z;
    wsum += w[j];
  }
  if (c->norm_topk)
    for (int j = 0; j < k; ++j) w[j] /= wsum;
  return ORC_OK;
}

// One expert's FFN on one token, direct-routed form (work log Parts 4 and 10):
//   gu[r] = sum_h x[h] * W13e[r, h],  r < 2*inter  (gate rows first, then up rows)
//   a[i]  = silu(gu[i]) * gu[inter + i]
//   y[h]  = sum_i W2e[h, i] * a[i]
static void expert_ffn(int H, int inter, int32_t dtype, const uint16_t* x,
                       const uint16_t* w13e, const uint16_t* w2e, double* y) {
  std::vector<double> gu(2 * static_cast<size_t>(inter));
  for (int r = 0; r < 2 * inter; ++r) {
    double acc = 0.0;
    for (int h = 0; h < H; ++h)
      acc += decode(x[h], dtype) * decode(w13e[static_cast<size_t>(r) * H + h], dtype);
    gu[r] = acc;
  }
  std::vector<double> a(inter);
  for (int i = 0; i < inter; ++i) a[i] = silu(gu[i]) * gu[inter + i];
  for (int h = 0; h < H; ++h) {
    double acc = 0.0;
    for (int i = 0; i < inter; ++i)
      acc += decode(w2e[static_cast<size_t>(h) * inter + i], dtype) * a[i];
    y[h] = acc;
  }
}

// The whole block for T independent tokens, direct-routed formulation.
//   x        [T, H]           token activations
//   wr       [E, H]           router (gate) weights
//   w13_e    E pointers, each [2I, H] (may be NULL for experts no token selects)
//   w2_e     E pointers, each [H, I]
//   sw13     [2Is, H] or NULL, sw2 [H, Is] or NULL, swg [H] or NULL
// Outputs: ids [T, k], w [T, k], logits [T, E] (may be NULL), out [T, H].
//   out[t, h] = sum_j w[t, j] * y_{ids[t, j]}[h]  +  g_t * ys[h]
int oracle_moe_forward(const oracle_cfg* c, int32_t T, const uint16_t* x, const uint16_t* wr,
                       const uint16_t* const* w13_e, const uint16_t* const* w2_e,
                       const uint16_t* sw13, const uint16_t* sw2, const uint16_t* swg,
                       int32_t* ids, double* w, double* logits, double* out) {
  if (!cfg_ok(c) || T < 0 || !x || !wr || !w13_e || !w2_e || !ids || !w || !out)
    return ORC_BAD_ARG;
  if (c->shared_inter > 0 && (!sw13 || !sw2)) return ORC_BAD_ARG;
  if (c->has_shared_gate && (!swg || c->shared_inter == 0)) return ORC_BAD_ARG;
  const int H = c->hidden, E = c->n_experts, k = c->top_k, I = c->inter;
  std::vector<double> lg(E), y(H), ys(H);
  for (int t = 0; t < T; ++t) {
    const uint16_t* xt = x + static_cast<size_t>(t) * H;
    int32_t* idt = ids + static_cast<size_t>(t) * k;
    double* wt = w + static_cast<size_t>(t) * k;
    int rc = oracle_router_token(c, xt, wr, lg.data(), idt, wt);
    if (rc) return rc;
    if (logits)
      for (int e = 0; e < E; ++e) logits[static_cast<size_t>(t) * E + e] = lg[e];
    double* ot = out + static_cast<size_t>(t) * H;
    for (int h = 0; h < H; ++h) ot[h] = 0.0;
    for (int j = 0; j < k; ++j) {
      const int e = idt[j];
      if (!w13_e[e] || !w2_e[e]) return ORC_MISSING_EXPERT;
      expert_ffn(H, I, c->dtype, xt, w13_e[e], w2_e[e], y.data());
      for (int h = 0; h < H; ++h) ot[h] += wt[j] * y[h];
    }
    if (c->shared_inter > 0) {
      expert_ffn(H, c->shared_inter, c->dtype, xt, sw13, sw2, ys.data());
      double g = 1.0;
      if (c->has_shared_gate) {
        double s = 0.0;
        for (int h = 0; h < H; ++h) s += decode(xt[h], c->dtype) * decode(swg[h], c->dtype);
        g = sigmoid(s);
      }
      for (int h = 0; h < H; ++h) ot[h] += g * ys[h];
    }
  }
  return ORC_OK;
}

// The same block in the fallback formulation of the work log's Part 3, kept
// as a separately written second formulation: copy the selected experts'
// weights out (index_select), run one dense linear over the k*2I stacked rows,
// SiluAndMul on the [k, 2I] view, a batched [k,1,I] x [k,I,H] product, then the
// weighted sum; the shared expert runs as its own gate_up / SiluAndMul / down.
int oracle_moe_forward_gather(const oracle_cfg* c, int32_t T, const uint16_t* x,
                              const uint16_t* wr, const uint16_t* const* w13_e,
                              const uint16_t* const* w2_e, const uint16_t* sw13,
                              const uint16_t* sw2, const uint16_t* swg, double* out) {
  if (!cfg_ok(c) || T < 0 || !x || !wr || !w13_e || !w2_e || !out) return ORC_BAD_ARG;
  if (c->shared_inter > 0 && (!sw13 || !sw2)) return ORC_BAD_ARG;
  if (c->has_shared_gate && (!swg || c->shared_inter == 0)) return ORC_BAD_ARG;
  const size_t H = c->hidden, E = c->n_experts, k = c->top_k, I = c->inter;
  const size_t Is = c->shared_inter;
  std::vector<double> lg(E), wk(k);
  std::vector<int32_t> idk(k);
  for (int32_t t = 0; t < T; ++t) {
    const uint16_t* xt = x + static_cast<size_t>(t) * H;
    int rc = oracle_router_token(c, xt, wr, lg.data(), idk.data(), wk.data());
    if (rc) return rc;
    // index_select: materialise W13s[k, 2I, H] and W2s[k, H, I] as doubles.
    std::vector<double> w13s(k * 2 * I * H), w2s(k * H * I), xd(H);
    for (size_t j = 0; j < k; ++j) {
      const uint16_t* a = w13_e[idk[j]];
      const uint16_t* b = w2_e[idk[j]];
      if (!a || !b) return ORC_MISSING_EXPERT;
      for (size_t q = 0; q < 2 * I * H; ++q) w13s[j * 2 * I * H + q] = decode(a[q], c->dtype);
      for (size_t q = 0; q < H * I; ++q) w2s[j * H * I + q] = decode(b[q], c->dtype);
    }
    for (size_t h = 0; h < H; ++h) xd[h] = decode(xt[h], c->dtype);
    // F.linear(x, W13s.view(k*2I, H)) -> [k*2I]
    std::vector<double> flat(k * 2 * I);
    for (size_t r = 0; r < k * 2 * I; ++r) {
      double acc = 0.0;
      for (size_t h = 0; h < H; ++h) acc += xd[h] * w13s[r * H + h];
      flat[r] = acc;
    }
    // view [k, 2I] -> SiluAndMul -> act [k, I]
    std::vector<double> act(k * I);
    for (size_t j = 0; j < k; ++j)
      for (size_t i = 0; i < I; ++i)
        act[j * I + i] = silu(flat[j * 2 * I + i]) * flat[j * 2 * I + I + i];
    // bmm: [k,1,I] x [k,I,H] where the [I,H] operand is W2s[j] transposed.
    std::vector<double> yk(k * H);
    for (size_t j = 0; j < k; ++j)
      for (size_t h = 0; h < H; ++h) {
        double acc = 0.0;
        for (size_t i = 0; i < I; ++i) acc += act[j * I + i] * w2s[j * H * I + h * I + i];
        yk[j * H + h] = acc;
      }
    // weighted sum over the k experts.
    double* ot = out + static_cast<size_t>(t) * H;
    for (size_t h = 0; h < H; ++h) {
      double acc = 0.0;
      for (size_t j = 0; j < k; ++j) acc += wk[j] * yk[j * H + h];
      ot[h] = acc;
    }
    // shared expert: gate_up, SiluAndMul, down (+ optional sigmoid gate).
    if (Is > 0) {
      std::vector<double> sgu(2 * Is), sact(Is);
      for (size_t r = 0; r < 2 * Is; ++r) {
        double acc = 0.0;
        for (size_t h = 0; h < H; ++h) acc += xd[h] * decode(sw13[r * H + h], c->dtype);
        sgu[r] = acc;
      }
      for (size_t i = 0; i < Is; ++i) sact[i] = silu(sgu[i]) * sgu[Is + i];
      double g = 1.0;
      if (c->has_shared_gate) {
        double s = 0.0;
        for (size_t h = 0; h < H; ++h) s += xd[h] * decode(swg[h], c->dtype);
        g = sigmoid(s);
      }
      for (size_t h = 0; h < H; ++h) {
        double acc = 0.0;
        for (size_t i = 0; i < Is; ++i) acc += decode(sw2[h * Is + i], c->dtype) * sact[i];
        ot[h] += g * acc;
      }
    }
  }
  return ORC_OK;
}

// Stage entry for the pages' known-data check (work log Part 1): the W2 dot
// products and the routing-weighted combine, given the activation directly.
//   out[h] = sum_j w[j] * sum_i W2[ids[j], h, i] * act[j, i]
int oracle_w2_combine(const oracle_cfg* c, const double* act, const int32_t* ids,
                      const double* w, const uint16_t* const* w2_e, double* out) {
  if (!cfg_ok(c) || !act || !ids || !w || !w2_e || !out) return ORC_BAD_ARG;
  const int H = c->hidden, k = c->top_k, I = c->inter;
  for (int h = 0; h < H; ++h) out[h] = 0.0;
  for (int j = 0; j < k; ++j) {
    if (ids[j] < 0 || ids[j] >= c->n_experts) return ORC_BAD_ARG;
    const uint16_t* b = w2_e[ids[j]];
    if (!b) return ORC_MISSING_EXPERT;
    for (int h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int i = 0; i < I; ++i)
        acc += decode(b[static_cast<size_t>(h) * I + i], c->dtype) * act[static_cast<size_t>(j) * I + i];
      out[h] += w[j] * acc;
    }
  }
  return ORC_OK;
}

}  // extern "C"
