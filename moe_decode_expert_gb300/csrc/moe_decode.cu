// moe_decode.cu — the whole T = 1 decode MoE block in one kernel launch.
//
// What it computes ("BI-V100 inference work log", Parts 3, 4, 9, 10):
// router GEMV + softmax + top-k, the direct-routed W13 GEMV that reads only
// the selected experts' rows in place (W13[expert_ids[k], row, :]) with
// SiluAndMul fused into it, the W2 GEMV W2[expert_ids[k], h, :] fused with
// the routing-weighted sum, and the shared expert (gate_up, SiluAndMul, down,
// optional sigmoid gate) fused into the same pass.
//
// How (GB300 design, not the pages' BI-V100 kernels): one CTA per SM, each
// owning a slice of every phase, all phases in one launch.
//   phase 1  routing-independent rows — router rows, the shared gate row and
//            the shared expert's gate/up pairs — as warp-per-row dot products
//            with 16-byte streaming loads issued before x lands in smem;
//            results are published as (value, epoch) exchange words.
//   phase 2  every CTA gathers the E logits (one L2 round trip when they are
//            all published), and one warp ranks them (fp32, lower index wins
//            ties) and forms the routing weights; no grid barrier and no
//            second kernel.
//   phase 3  thread 0 bulk-copies (TMA, untiled) the selected experts' W2
//            rows of this CTA's output slice into smem while the warps
//            compute this CTA's share of the k*I routed gate/up pairs
//            (W13 rows streamed to registers), apply SiLU*up and publish act.
//   phase 4  every CTA gathers all k*I + Is activations, waits for its W2
//            rows, and computes its slice of out[h] = sum_j w_j (W2_j act_j)
//            + g (Ws2 sact).
// The two exchanges replace two kernel boundaries; each wait is bounded by
// the GPU global timer and records an error instead of hanging.  The kernel
// triggers programmatic dependent launch at entry so the next call on the
// stream launches early and waits in its own prologue.

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kChunks = 8;  // 16-byte chunks per lane per row kept in flight

struct DecodeArgs {
  const uint8_t* x;
  const uint8_t* wr;
  const uint8_t* w13;
  const uint8_t* w2;
  const uint8_t* sw13;
  const uint8_t* sw2;
  const uint8_t* swg;
  int32_t* topk_ids;
  float* topk_w;
  void* out;
  Control* ctrl;
  uint64_t* ll_logits;
  uint64_t* ll_act;
  int H, E, k, I, Is, has_gate, norm_topk, out_dtype;
  int static_weights;  // MOE_FLAG_STATIC_WEIGHTS: weight reads may precede the PDL wait
  uint32_t off_lg, off_act, off_w2;
  uint64_t timeout_ns;
};

// Up to two weight rows of H 2-byte elements, streamed to registers 16 bytes
// per lane per chunk (lane-strided, so a warp reads 512 contiguous bytes per
// instruction), then dotted with x held in shared memory as fp32.
template <int DT>
struct RowPair {
  const uint8_t* r0;
  const uint8_t* r1;
  int two;   // 1: two rows, 0: one row
  uint4 v0[kChunks], v1[kChunks];

  __device__ __forceinline__ void issue(int base, int nch, int lane) {
#pragma unroll
    for (int t = 0; t < kChunks; ++t) {
      const int c = base + lane + 32 * t;
      const bool in = c < nch;
      v0[t] = in ? ld_stream16(r0 + 16 * static_cast<size_t>(c)) : make_uint4(0, 0, 0, 0);
      v1[t] = (in && two) ? ld_stream16(r1 + 16 * static_cast<size_t>(c)) : make_uint4(0, 0, 0, 0);
    }
  }

  // Completes the dot products whose first batch was issued with issue(0).
  __device__ __forceinline__ void finish(const float* xs, int nch, int lane, float& d0, float& d1) {
    float a0 = 0.f, a1 = 0.f;
    for (int base = 0; base < nch; base += 32 * kChunks) {
      if (base) issue(base, nch, lane);
#pragma unroll
      for (int t = 0; t < kChunks; ++t) {
        const int c = base + lane + 32 * t;
        if (c < nch) {
          const float4 xa = reinterpret_cast<const float4*>(xs)[2 * c];
          const float4 xb = reinterpret_cast<const float4*>(xs)[2 * c + 1];
          float f[8];
          unpack8<DT>(v0[t], f);
          a0 = fmaf(f[0], xa.x, a0); a0 = fmaf(f[1], xa.y, a0);
          a0 = fmaf(f[2], xa.z, a0); a0 = fmaf(f[3], xa.w, a0);
          a0 = fmaf(f[4], xb.x, a0); a0 = fmaf(f[5], xb.y, a0);
          a0 = fmaf(f[6], xb.z, a0); a0 = fmaf(f[7], xb.w, a0);
          if (two) {
            unpack8<DT>(v1[t], f);
            a1 = fmaf(f[0], xa.x, a1); a1 = fmaf(f[1], xa.y, a1);
            a1 = fmaf(f[2], xa.z, a1); a1 = fmaf(f[3], xa.w, a1);
            a1 = fmaf(f[4], xb.x, a1); a1 = fmaf(f[5], xb.y, a1);
            a1 = fmaf(f[6], xb.z, a1); a1 = fmaf(f[7], xb.w, a1);
          }
        }
      }
    }
    d0 = warp_sum(a0);
    d1 = warp_sum(a1);
  }
};

// DEPTH 1: one gate/up pair in flight per warp (<= 128 registers, two CTAs per
// SM fit); DEPTH 2: two pairs in flight (one CTA per SM), for configs with more
// routed pairs per CTA than warps.
template <int DT, int DEPTH>
__global__ void __launch_bounds__(kDecThreads, 3 - DEPTH) decode_fused_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_ids[32];
  __shared__ float s_sel[32];
  __shared__ float s_w[32];
  __shared__ float s_gate;
  __shared__ uint32_t s_epoch;
  __shared__ uint32_t s_fail;
  __shared__ int s_second_arrive_done;
  __shared__ volatile int s_ready[32];  // slot r ranked (its id is in s_ids[r])

  float* xs = reinterpret_cast<float*>(smem);
  float* lg = reinterpret_cast<float*>(smem + a.off_lg);
  float* acts = reinterpret_cast<float*>(smem + a.off_act);
  uint8_t* w2s = smem + a.off_w2;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x, G = gridDim.x;
  const int H = a.H, E = a.E, k = a.k, I = a.I, Is = a.Is;
  const int h0 = static_cast<int>((static_cast<long long>(H) * cta) / G);
  const int hn = static_cast<int>((static_cast<long long>(H) * (cta + 1)) / G) - h0;
  const size_t rowb = static_cast<size_t>(H) * 2;
  const int nch = H >> 3;

  if (tid == 0) {
    mbar_init(&bar, 2);
    mbar_fence_init();
    s_fail = 0;
    s_second_arrive_done = 0;
    for (int r = 0; r < 32; ++r) s_ready[r] = 0;
  }
  pdl_launch_dependents();
  __syncthreads();

  // ---- phase 1: routing-independent rows; the first round's loads go out
  // before x is staged (and, with static weights, before the PDL wait)
  const int n1 = E + a.has_gate + Is;
  int q = warp;
  int u = q * G + cta;
  RowPair<DT> rp;
  auto setup_unit = [&](int uu) {
    if (uu < E) {
      rp.r0 = a.wr + static_cast<size_t>(uu) * rowb; rp.r1 = rp.r0; rp.two = 0;
    } else if (uu < E + a.has_gate) {
      rp.r0 = a.swg; rp.r1 = rp.r0; rp.two = 0;
    } else {
      const int i = uu - E - a.has_gate;
      rp.r0 = a.sw13 + static_cast<size_t>(i) * rowb;
      rp.r1 = a.sw13 + static_cast<size_t>(Is + i) * rowb;
      rp.two = 1;
    }
  };
  auto issue_shared_w2 = [&]() {  // thread 0: the shared expert's W2 rows of this CTA's slice
    if (Is > 0 && hn > 0) {
      const uint32_t bytes = static_cast<uint32_t>(hn) * Is * 2;
      mbar_arrive_expect_tx(&bar, bytes);
      bulk_g2s(w2s + static_cast<size_t>(k) * hn * I * 2, a.sw2 + static_cast<size_t>(h0) * Is * 2, bytes, &bar);
    } else {
      mbar_arrive(&bar);
    }
  };
  if (a.static_weights) {
    if (u < n1) { setup_unit(u); rp.issue(0, nch, lane); }
    if (tid == 0) issue_shared_w2();
  }
  pdl_wait();  // x (and anything else an earlier kernel wrote) is visible from here
  if (!a.static_weights && u < n1) { setup_unit(u); rp.issue(0, nch, lane); }

  for (int c = tid; c < nch; c += kDecThreads) {
    float f[8];
    unpack8<DT>(ld_nc16(a.x + 16 * static_cast<size_t>(c)), f);
    reinterpret_cast<float4*>(xs)[2 * c] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(xs)[2 * c + 1] = make_float4(f[4], f[5], f[6], f[7]);
  }
  if (tid == 0) {
    uint32_t ep = ld_relaxed_u32(&a.ctrl->gen) + 1u;
    s_epoch = ep ? ep : 1u;
    // The arrival counter of the other parity was last used by the previous
    // launch, which has completed; clear it for the next launch.
    if (cta == 0) atomicExch(&a.ctrl->arrive[(s_epoch + 1u) & 1u], 0u);
    if (!a.static_weights) issue_shared_w2();
  }
  __syncthreads();
  const uint32_t epoch = s_epoch;

  while (u < n1) {
    float d0, d1;
    rp.finish(xs, nch, lane, d0, d1);
    if (lane == 0) {
      if (u < E + a.has_gate) ll_store(a.ll_logits + u, d0, epoch);
      else ll_store(a.ll_act + static_cast<size_t>(k) * I + (u - E - a.has_gate), silu_f(d0) * d1, epoch);
    }
    q += kDecWarps;
    u = q * G + cta;
    if (u < n1) { setup_unit(u); rp.issue(0, nch, lane); }
  }

  // ---- phase 2 (warp 0): gather the logits and rank them.  Each ranked
  // expert is published to the other warps, and its W2 rows requested, as
  // soon as its round ends, so expert loads overlap the rest of the ranking.
  if (warp == 0) {
    const int nl = E + a.has_gate;
    const bool ok = ll_gather(a.ll_logits, lg, nl, lane, 32, epoch, global_ns() + a.timeout_ns);
    if (__all_sync(0xffffffffu, ok)) {
      const uint32_t bytes = static_cast<uint32_t>(hn) * I * 2;
      if (lane == 0) {
        if (hn > 0) mbar_arrive_expect_tx(&bar, bytes * k);
        else mbar_arrive(&bar);
        s_second_arrive_done = 1;
      }
      __syncwarp();
      auto publish = [&](int r) {
        if (lane == 0) {
          __threadfence_block();
          s_ready[r] = 1;
        }
      };
      if (E <= 256) {
        warp_topk_sorted8(lg, E, k, s_ids, s_sel, publish);
      } else {
        warp_topk<32>(lg, E, k, s_ids, s_sel);
        __syncwarp();
        for (int r = 0; r < k; ++r) publish(r);
      }
      __syncwarp();
      // this CTA's W2 rows of the k experts, one lane per expert
      if (hn > 0 && lane < k)
        bulk_g2s(w2s + static_cast<size_t>(lane) * hn * I * 2,
                 a.w2 + (static_cast<size_t>(s_ids[lane]) * H + h0) * I * 2, bytes, &bar);
      warp_routing_weights(lg, E, s_sel, k, a.norm_topk, s_w);
      if (lane == 0) s_gate = a.has_gate ? sigmoid_f(lg[E]) : 1.0f;
      __syncwarp();
      if (cta == 0 && lane < k) {
        a.topk_ids[lane] = s_ids[lane];
        a.topk_w[lane] = s_w[lane];
      }
    } else if (lane == 0) {
      s_fail = kDevTimeoutLogits;
      __threadfence_block();
      for (int r = 0; r < 32; ++r) s_ready[r] = 1;  // let the waiting warps see the failure
    }
  }

  // ---- phase 3: this CTA's share of the k*I routed gate/up pairs; a warp
  // starts a pair as soon as the pair's expert has been ranked.  With
  // DEPTH == 2 a warp keeps two pairs' rows in flight at once.
  const int P = k * I;
  auto wait_slot = [&](int j) -> bool {
    const uint64_t deadline = global_ns() + a.timeout_ns;
    while (s_ready[j] == 0) {
      if (global_ns() > deadline) return false;
      __nanosleep(32);
    }
    __threadfence_block();
    return true;
  };
  auto start_pair = [&](RowPair<DT>& r, int p) -> bool {
    const int j = p / I, i = p - j * I;
    if (!wait_slot(j)) {
      if (lane == 0) s_fail = kDevTimeoutLogits;
      return false;
    }
    if (s_fail) return false;
    const size_t erow = static_cast<size_t>(s_ids[j]) * 2 * I;
    r.r0 = a.w13 + (erow + i) * rowb;
    r.r1 = a.w13 + (erow + I + i) * rowb;
    r.two = 1;
    r.issue(0, nch, lane);
    return true;
  };
  auto end_pair = [&](RowPair<DT>& r, int p) {
    float g, up;
    r.finish(xs, nch, lane, g, up);
    if (lane == 0) ll_store(a.ll_act + p, silu_f(g) * up, epoch);
  };
  if constexpr (DEPTH == 2) {
    RowPair<DT> rq;
    for (int qq = warp;; qq += 2 * kDecWarps) {
      const int pa = qq * G + cta, pb = (qq + kDecWarps) * G + cta;
      if (pa >= P) break;
      if (!start_pair(rp, pa)) break;
      const bool has_b = pb < P && start_pair(rq, pb);
      end_pair(rp, pa);
      if (!has_b) break;
      end_pair(rq, pb);
    }
  } else {
    for (int qq = warp;; qq += kDecWarps) {
      const int p = qq * G + cta;
      if (p >= P) break;
      if (!start_pair(rp, p)) break;
      end_pair(rp, p);
    }
  }

  {
    // ---- phase 4: all activations, this CTA's W2 rows, out slice
    // One thread per CTA counts CTAs in and waits for all G of them; only then
    // do all threads read the exchange words (one pass when they have landed;
    // the epoch tags still catch any word not yet visible).  Polling the words
    // themselves from every thread of every CTA congests the L2 lines they
    // live in and delays the producers' stores.
    __syncthreads();
    bool ok = true;
    if (tid == 0 && !s_fail) {
      uint32_t* cnt = &a.ctrl->arrive[epoch & 1u];
      atomicAdd(cnt, 1u);
      const uint64_t deadline = global_ns() + a.timeout_ns;
      while (ld_relaxed_u32(cnt) < static_cast<uint32_t>(G)) {
        if (global_ns() > deadline) { ok = false; break; }
      }
      if (!ok) s_fail = kDevTimeoutAct;
    }
    __syncthreads();
    if (!s_fail) ok = ll_gather(a.ll_act, acts, P + Is, tid, kDecThreads, epoch, global_ns() + a.timeout_ns);
    if (!ok) s_fail = kDevTimeoutAct;
    if (tid == 0 && !mbar_wait_until(&bar, 0, global_ns() + a.timeout_ns)) s_fail = kDevTimeoutCopy;
    __syncthreads();
    if (!s_fail) {
      // Fold the routing weight (and the shared gate) into the activations,
      // so each output is one dot product over the concatenated
      // [k*I routed | Is shared] activation vector.  Integer quotients come
      // from an fp32 reciprocal, exact for indices below 2^22.
      const float inv_I = 1.0f / static_cast<float>(I);
      for (int i = tid; i < P + Is; i += kDecThreads) {
        const int j = i < P ? __float2int_rz((static_cast<float>(i) + 0.5f) * inv_I) : k;
        acts[i] *= j < k ? s_w[j] : s_gate;
      }
      __syncthreads();
      // Two output rows per warp, 16 threads per row; thread tl takes chunks
      // tl, tl+16, ... (16-byte chunks of 8 weights) into four independent
      // accumulators.  The loop bound is warp-uniform so every lane reaches the
      // shuffles.
      const int cpe = I >> 3;
      const int nchunk = (P + Is) >> 3;
      const float inv_cpe = 1.0f / static_cast<float>(cpe);
      const int tl = tid & 15;
      for (int rbase = warp * 2; rbase < hn; rbase += kDecThreads / 16) {
        const int r = rbase + ((tid >> 4) & 1);
        const bool active = r < hn;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (active) {
          const uint8_t* rrow = w2s + static_cast<size_t>(r) * I * 2;
          const uint8_t* srow = w2s + (static_cast<size_t>(k) * hn * I + static_cast<size_t>(r) * Is) * 2;
          for (int c0 = tl; c0 < nchunk; c0 += 64) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int c = c0 + 16 * u;
              if (c < nchunk) {
                const int j = __float2int_rz((static_cast<float>(c) + 0.5f) * inv_cpe);
                const uint8_t* wp = j < k ? rrow + (static_cast<size_t>(j) * hn * I + (c - j * cpe) * 8) * 2
                                          : srow + static_cast<size_t>(c - k * cpe) * 16;
                const uint4 v = *reinterpret_cast<const uint4*>(wp);
                const float4 xa = reinterpret_cast<const float4*>(acts)[2 * c];
                const float4 xb = reinterpret_cast<const float4*>(acts)[2 * c + 1];
                float f[8];
                unpack8<DT>(v, f);
                float t = f[0] * xa.x;
                t = fmaf(f[1], xa.y, t); t = fmaf(f[2], xa.z, t); t = fmaf(f[3], xa.w, t);
                t = fmaf(f[4], xb.x, t); t = fmaf(f[5], xb.y, t); t = fmaf(f[6], xb.z, t);
                t = fmaf(f[7], xb.w, t);
                acc[u] += t;
              }
            }
          }
        }
        float sum = (acc[0] + acc[1]) + (acc[2] + acc[3]);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (active && tl == 0) store_out(a.out, h0 + r, sum, a.out_dtype);
      }
      // Every CTA has read the epoch before publishing its activations and CTA 0
      // has now seen all of them, so the next launch may use the next epoch.
      if (cta == 0 && tid == 0) atomicExch(&a.ctrl->gen, epoch);
      return;
    }
  }

  // ---- failure path: record, let this CTA's own bulk copies land, bump the epoch
  if (tid == 0) {
    report_error(a.ctrl, s_fail, static_cast<uint32_t>(cta));
    if (!s_second_arrive_done) mbar_arrive(&bar);
    mbar_wait_until(&bar, 0, global_ns() + a.timeout_ns);
    if (cta == 0) atomicExch(&a.ctrl->gen, epoch);
  }
}

// ------------------------------------------------------------------ host side
int decode_grid(const moe_cfg_t& c) {
  // One CTA per SM; never more CTAs than routed pairs, so that every CTA
  // publishes at least one activation (the epoch hand-over relies on it).
  const int pairs = c.top_k * c.inter;
  int g = sm_count();
  if (g > pairs) g = pairs;
  return g < 1 ? 1 : g;
}

static void decode_smem_layout(const moe_cfg_t& c, int G, uint32_t& off_lg, uint32_t& off_act,
                               uint32_t& off_w2, size_t& total) {
  const size_t H = c.hidden, E = c.n_experts, k = c.top_k, I = c.inter, Is = c.shared_inter;
  const size_t hn_max = (H + G - 1) / G;
  size_t off = align_up(H * 4, 128);
  off_lg = static_cast<uint32_t>(off);
  off += align_up((E + 2) * 4, 128);
  off_act = static_cast<uint32_t>(off);
  off += align_up((k * I + Is + 2) * 4, 128);
  off_w2 = static_cast<uint32_t>(off);
  off += align_up(hn_max * (k * I + Is) * 2, 128);
  total = off;
}

size_t decode_smem_bytes(const moe_cfg_t& c, int G) {
  uint32_t a, b, d;
  size_t t;
  decode_smem_layout(c, G, a, b, d, t);
  return t;
}

template <int DT, int DEPTH>
static moe_status_t launch_decode_dt(const DecodeArgs& args, int G, size_t smem, cudaStream_t st) {
  static int configured_dev = -1;
  static size_t configured_smem = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev || configured_smem < smem) {
    if (cudaFuncSetAttribute(decode_fused_kernel<DT, DEPTH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return check_launch("cudaFuncSetAttribute(decode)");
    configured_dev = dev;
    configured_smem = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, decode_fused_kernel<DT, DEPTH>, args) != cudaSuccess)
    return check_launch("decode_fused_kernel");
  stat_kernels(1);
  return MOE_OK;
}

moe_status_t launch_decode_fused(const moe_cfg_t& c, const BlockPtrs& p, uint8_t* ws,
                                 const WsLayout& L, cudaStream_t st) {
  const int G = decode_grid(c);
  DecodeArgs a;
  a.x = static_cast<const uint8_t*>(p.x);
  a.wr = static_cast<const uint8_t*>(p.router_w);
  a.w13 = static_cast<const uint8_t*>(p.w13);
  a.w2 = static_cast<const uint8_t*>(p.w2);
  a.sw13 = static_cast<const uint8_t*>(p.shared_w13);
  a.sw2 = static_cast<const uint8_t*>(p.shared_w2);
  a.swg = static_cast<const uint8_t*>(p.shared_gate_w);
  a.topk_ids = p.topk_ids;
  a.topk_w = p.topk_w;
  a.out = p.out;
  a.ctrl = reinterpret_cast<Control*>(ws + L.ctrl);
  a.ll_logits = reinterpret_cast<uint64_t*>(ws + L.ll_logits);
  a.ll_act = reinterpret_cast<uint64_t*>(ws + L.ll_act);
  a.H = c.hidden; a.E = c.n_experts; a.k = c.top_k; a.I = c.inter; a.Is = c.shared_inter;
  a.has_gate = c.has_shared_gate; a.norm_topk = c.norm_topk; a.out_dtype = c.out_dtype;
  a.static_weights = (c.flags & MOE_FLAG_STATIC_WEIGHTS) ? 1 : 0;
  size_t smem;
  decode_smem_layout(c, G, a.off_lg, a.off_act, a.off_w2, smem);
  a.timeout_ns = wait_timeout_ns();
  if (smem > 227 * 1024)
    return set_error(MOE_ERR_UNSUPPORTED, "decode: needs %zu B of shared memory per CTA (max 232448)", smem);
  // two pairs in flight per warp when a CTA has more routed pairs than warps
  const bool deep = (c.top_k * c.inter + G - 1) / G > kDecWarps;
  if (c.dtype == MOE_BF16)
    return deep ? launch_decode_dt<MOE_BF16, 2>(a, G, smem, st) : launch_decode_dt<MOE_BF16, 1>(a, G, smem, st);
  return deep ? launch_decode_dt<MOE_F16, 2>(a, G, smem, st) : launch_decode_dt<MOE_F16, 1>(a, G, smem, st);
}

}  // namespace moe
