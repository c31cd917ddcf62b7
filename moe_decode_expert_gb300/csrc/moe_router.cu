// moe_router.cu — router GEMV/GEMM, fp32 softmax and top-k for T >= 1 tokens.
//
// "BI-V100 inference work log", Part 3 (gate, topk, softmax of the fallback
// path) and Part 8 (the separate topk and softmax launches it counts);
// "Decode throughput analysis report", code-level profiling section (the
// fused topk_softmax kernel is missing on the pages' hardware).
//
// Two launches: a tiled fp32 GEMM logits[T, E(+1)] = x[T, H] . Wr^T (column E
// is the shared-expert gate logit x . wg when there is one), then one warp
// per token ranks the E logits (fp32 key, lower index first on ties) and
// writes ids, routing weights and (optionally) the raw logits.

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_stages.cuh"

namespace moe {

constexpr int kRBM = 64;   // router rows (experts) per CTA tile
constexpr int kRBN = 64;   // tokens per CTA tile
constexpr int kRBK = 32;   // hidden elements per k-step
constexpr int kRouterGemvMaxT = 64;  // T up to this uses the row-per-warp kernel

template <int DT>
__global__ void __launch_bounds__(256) router_logits_kernel(const uint8_t* x,
                                                            const uint8_t* wr,
                                                            const uint8_t* swg, int T,
                                                            int H, int E, int E1, float* __restrict__ logits) {
  pdl_launch_dependents();  // let the next kernel on the stream launch early
  pdl_wait();               // inputs written by the previous kernel are visible
  __shared__ float As[kRBK][kRBM + 4];   // router rows, k-major
  __shared__ float Bs[kRBK][kRBN + 4];   // tokens, k-major
  const int tid = threadIdx.x;
  const int m0 = blockIdx.x * kRBM, n0 = blockIdx.y * kRBN;
  const int ty = tid >> 4, tx = tid & 15;
  const size_t rowb = static_cast<size_t>(H) * 2;
  // each thread stages one 16-byte chunk (8 elements) of each tile per k-step
  const int lr = tid >> 2, lk = (tid & 3) * 8;
  const int e = m0 + lr, t = n0 + lr;
  const uint8_t* arow = nullptr;
  if (e < E) arow = wr + static_cast<size_t>(e) * rowb;
  else if (e == E && E1 > E) arow = swg;
  const uint8_t* brow = t < T ? x + static_cast<size_t>(t) * rowb : nullptr;

  float acc[4][4] = {};
  for (int k0 = 0; k0 < H; k0 += kRBK) {
    float fa[8], fb[8];
    const bool kin = k0 + lk < H;   // H % 8 == 0, so a chunk is all in or all out
    if (arow && kin) unpack8<DT>(ld_nc16(arow + 2 * static_cast<size_t>(k0 + lk)), fa);
    else for (int i = 0; i < 8; ++i) fa[i] = 0.f;
    if (brow && kin) unpack8<DT>(ld_nc16(brow + 2 * static_cast<size_t>(k0 + lk)), fb);
    else for (int i = 0; i < 8; ++i) fb[i] = 0.f;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      As[lk + i][lr] = fa[i];
      Bs[lk + i][lr] = fb[i];
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kRBK; ++kk) {
      const float4 av = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 bv = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float ar[4] = {av.x, av.y, av.z, av.w};
      const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int ee = m0 + ty * 4 + i, tt = n0 + tx * 4 + j;
      if (ee < E1 && tt < T) logits[static_cast<size_t>(tt) * E1 + ee] = acc[i][j];
    }
}

// Small T: one warp per router row (held in registers as fp32, 2048 columns
// per pass), dotted with a tile of up to 16 tokens staged in shared memory as
// fp32.  Grid (ceil(E1 / 8), ceil(T / 16)).
constexpr int kGvTok = 16;
template <int DT>
__global__ void __launch_bounds__(256) router_gemv_kernel(const uint8_t* x,
                                                          const uint8_t* wr,
                                                          const uint8_t* swg, int T, int H, int E,
                                                          int E1, float* __restrict__ logits) {
  pdl_launch_dependents();  // let the next kernel on the stream launch early
  pdl_wait();               // inputs written by the previous kernel are visible
  extern __shared__ __align__(16) float xt[];  // [kGvTok][min(H, 2048)] fp32
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  const int t0 = blockIdx.y * kGvTok;
  const int nt = min(kGvTok, T - t0);
  const size_t rowb = static_cast<size_t>(H) * 2;
  const uint8_t* row = nullptr;
  if (e < E) row = wr + static_cast<size_t>(e) * rowb;
  else if (e == E && E1 > E) row = swg;
  float acc[kGvTok];
#pragma unroll
  for (int t = 0; t < kGvTok; ++t) acc[t] = 0.f;
  for (int k0 = 0; k0 < H; k0 += 2048) {
    const int kw = min(2048, H - k0);
    const int nch = kw >> 3;
    __syncthreads();
    // 8 loads in flight per thread before any is used (the tile is up to 16 x 2048).
    for (int base = threadIdx.x; base < nt * nch; base += 256 * 8) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int idx = base + 256 * u;
        if (idx < nt * nch) {
          const int t = idx / nch, c = idx - t * nch;
          v[u] = ld_nc16(x + (static_cast<size_t>(t0 + t) * H + k0 + 8 * c) * 2);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int idx = base + 256 * u;
        if (idx < nt * nch) {
          const int t = idx / nch, c = idx - t * nch;
          float f[8];
          unpack8<DT>(v[u], f);
          float4* d = reinterpret_cast<float4*>(xt + static_cast<size_t>(t) * 2048 + 8 * c);
          d[0] = make_float4(f[0], f[1], f[2], f[3]);
          d[1] = make_float4(f[4], f[5], f[6], f[7]);
        }
      }
    }
    __syncthreads();
    if (row) {
      float w[8][8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int c = lane + 32 * q;
        if (c < nch) unpack8<DT>(ld_stream16(row + (static_cast<size_t>(k0) + 8 * c) * 2), w[q]);
        else
#pragma unroll
          for (int i = 0; i < 8; ++i) w[q][i] = 0.f;
      }
#pragma unroll
      for (int t = 0; t < kGvTok; ++t) {
        if (t < nt) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int c = lane + 32 * q;
            if (c < nch) {
              const float4 a = reinterpret_cast<const float4*>(xt + static_cast<size_t>(t) * 2048)[2 * c];
              const float4 b = reinterpret_cast<const float4*>(xt + static_cast<size_t>(t) * 2048)[2 * c + 1];
              acc[t] = fmaf(w[q][0], a.x, acc[t]); acc[t] = fmaf(w[q][1], a.y, acc[t]);
              acc[t] = fmaf(w[q][2], a.z, acc[t]); acc[t] = fmaf(w[q][3], a.w, acc[t]);
              acc[t] = fmaf(w[q][4], b.x, acc[t]); acc[t] = fmaf(w[q][5], b.y, acc[t]);
              acc[t] = fmaf(w[q][6], b.z, acc[t]); acc[t] = fmaf(w[q][7], b.w, acc[t]);
            }
          }
        }
      }
    }
  }
  if (!row) return;
#pragma unroll
  for (int t = 0; t < kGvTok; ++t) {
    const float v = warp_sum(acc[t]);
    if (lane == 0 && t < nt) logits[static_cast<size_t>(t0 + t) * E1 + e] = v;
  }
}

// ---- small-T router on m16n8k16 tensor-core steps
// logits[t, e] for T <= 64 tokens and E + gate <= 257 rows: 16 router rows
// (the gate vector as row E) are the A operand, the tokens (8 per n-tile) the
// B columns.  CTA (m-tile, split s) takes columns [s*cpc, (s+1)*cpc) of H, its
// 8 warps 32-column chunks of that range; lane (g, t) streams 16-byte chunks
// of rows g and g + 8 and of token g (elements 0-3 of a chunk form one k-step,
// 4-7 the next, the same on both sides).  The warps' sums meet in shared
// memory and the CTA writes partial logits part[s][t][e]; the top-k kernel
// adds the splits in order.
template <int DT>
__global__ void __launch_bounds__(256) router_mma_kernel(const uint8_t* x,
                                                         const uint8_t* wr,
                                                         const uint8_t* swg, int T, int H, int E,
                                                         int E1, int cpc, float* __restrict__ part) {
  pdl_launch_dependents();  // let the next kernel on the stream launch early
  pdl_wait();               // inputs written by the previous kernel are visible
  __shared__ float red[8][16][64];  // [warp][row][token]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int m0 = blockIdx.x * 16, s = blockIdx.y;
  const int c0 = s * cpc, c1 = min(c0 + cpc, H);
  const size_t rowb = static_cast<size_t>(H) * 2;
  auto rowp = [&](int r) -> const uint8_t* {  // rows past E1 repeat the last row (discarded)
    const int e = min(m0 + r, E1 - 1);
    return e < E ? wr + static_cast<size_t>(e) * rowb : swg;
  };
  const uint8_t* ra = rowp(g);
  const uint8_t* rb = rowp(g + 8);
  const int nT = (T + 7) >> 3;
  float acc[8][4];
#pragma unroll
  for (int n = 0; n < 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;
  for (int cc = c0 + 32 * warp; cc < c1; cc += 256) {
    const bool cin = cc + 8 * t < c1;
    const int c = cin ? cc + 8 * t : c1 - 8;  // clamped: its B entries are zeroed
    const uint4 wa = ld_nc16(ra + 2 * static_cast<size_t>(c));
    const uint4 wb = ld_nc16(rb + 2 * static_cast<size_t>(c));
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      if (n < nT) {
        const int tok = min(n * 8 + g, T - 1);  // tokens past T repeat the last (discarded)
        uint4 xv = ld_nc16(x + (static_cast<size_t>(tok) * H + c) * 2);
        xv = cin ? xv : make_uint4(0u, 0u, 0u, 0u);
        mma16816<DT>(acc[n], wa.x, wb.x, wa.y, wb.y, xv.x, xv.y);
        mma16816<DT>(acc[n], wa.z, wb.z, wa.w, wb.w, xv.z, xv.w);
      }
    }
  }
  // D fragment: rows g / g + 8, tokens n*8 + 2t, 2t + 1
#pragma unroll
  for (int n = 0; n < 8; ++n) {
    if (n < nT) {
      red[warp][g][n * 8 + 2 * t] = acc[n][0];
      red[warp][g][n * 8 + 2 * t + 1] = acc[n][1];
      red[warp][g + 8][n * 8 + 2 * t] = acc[n][2];
      red[warp][g + 8][n * 8 + 2 * t + 1] = acc[n][3];
    }
  }
  __syncthreads();
  for (int i = tid; i < 16 * 64; i += 256) {
    const int r = i >> 6, tt = i & 63;
    const int e = m0 + r;
    if (tt < T && e < E1) {
      float v = 0.0f;
#pragma unroll
      for (int w = 0; w < 8; ++w) v += red[w][r][tt];
      part[(static_cast<size_t>(s) * T + tt) * E1 + e] = v;
    }
  }
}

// One warp per token: rank, weights, outputs.
// With nsplit > 0 the logits arrive as nsplit partial sums part[s][t][e]
// (router_mma_kernel): they are added in split order, stored into `logits`
// (the [T, E1] buffer later kernels read) and ranked from shared memory.
// One warp per token: rank, weights, outputs.
// With cnt != NULL each pair also takes its rank within its expert from a
// global counter per expert (the order within an expert is arbitrary).
template <int MAXM>
__global__ void __launch_bounds__(256) router_topk_kernel(float* logits, const float* part,
                                                          int nsplit, int T, int E, int E1, int k, int norm_topk,
                                                          int32_t* ids, float* w, float* logits_out, int32_t* cnt,
                                                          int32_t* rank) {
  pdl_launch_dependents();  // let the next kernel on the stream launch early
  pdl_wait();               // inputs written by the previous kernel are visible
  __shared__ int s_ids[8][32];
  __shared__ float s_sel[8][32];
  __shared__ float s_w[8][32];
  __shared__ float s_row[8][MAXM == 8 ? 258 : 1];
  const int warp = threadIdx.x >> 5;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  topk_token_stage<MAXM>(logits, part, nsplit, t, T, E, E1, k, norm_topk, ids, w, logits_out, s_ids[warp],
                         s_sel[warp], s_w[warp], s_row[warp]);
  if (cnt && (threadIdx.x & 31) < k) {
    const int e = s_ids[warp][threadIdx.x & 31];
    if (e >= 0 && e < E) rank[static_cast<size_t>(t) * k + (threadIdx.x & 31)] = atomicAdd(&cnt[e], 1);
  }
}

moe_status_t launch_router(const moe_cfg_t& c, const void* x, const void* router_w,
                           const void* shared_gate_w, int32_t T, int32_t* ids, float* w,
                           float* logits_out, uint8_t* ws, const WsLayout& L, cudaStream_t st,
                           int* nsplit_out, int32_t* cnt, int32_t* rank) {
  const int E = c.n_experts;
  const int E1 = E + 1;
  float* lg = reinterpret_cast<float*>(ws + L.r_logits);
  const uint8_t* swg = c.has_shared_gate ? static_cast<const uint8_t*>(shared_gate_w) : nullptr;
  const int stride = swg ? E1 : E;
  const uint8_t* xb = static_cast<const uint8_t*>(x);
  const uint8_t* wb = static_cast<const uint8_t*>(router_w);
  const bool tc = T >= kRouterTcMinT && tc_router_supported(c);
  int nsplit = 0;  // > 0: the logits are split partial sums (router_mma_kernel)
  if (tc) {
    float* part = L.r_part_splits ? reinterpret_cast<float*>(ws + L.r_part) : nullptr;
    if (moe_status_t s = launch_tc_router(c, x, router_w, swg, T, lg, part, stride,
                                          reinterpret_cast<Control*>(ws + L.ctrl), st, &nsplit))
      return s;
  } else if (T <= kRouterGemvMaxT && E1 <= 257 && c.hidden % 8 == 0) {
    const int nm = (stride + 15) / 16;
    int S = c.hidden / 256;
    const int smax = sm_count() / nm;
    if (S > smax) S = smax;
    if (S < 1) S = 1;
    const int cpc = ((c.hidden + S - 1) / S + 31) / 32 * 32;
    S = (c.hidden + cpc - 1) / cpc;
    float* part = reinterpret_cast<float*>(ws + L.r_part);
    if (c.dtype == MOE_BF16)
      launch_pdl(router_mma_kernel<MOE_BF16>, dim3(nm, S), dim3(256), 0, st, xb, wb, swg, T, c.hidden, E, stride, cpc, part);
    else
      launch_pdl(router_mma_kernel<MOE_F16>, dim3(nm, S), dim3(256), 0, st, xb, wb, swg, T, c.hidden, E, stride, cpc, part);
    nsplit = S;
  } else if (T <= kRouterGemvMaxT) {
    dim3 gg((E1 + 7) / 8, (T + kGvTok - 1) / kGvTok);
    const size_t sm = static_cast<size_t>(kGvTok) * 2048 * 4;
    if (c.dtype == MOE_BF16) {
      cudaFuncSetAttribute(router_gemv_kernel<MOE_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
      launch_pdl(router_gemv_kernel<MOE_BF16>, dim3(gg), dim3(256), sm, st, xb, wb, swg, T, c.hidden, E, stride, lg);
    } else {
      cudaFuncSetAttribute(router_gemv_kernel<MOE_F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
      launch_pdl(router_gemv_kernel<MOE_F16>, dim3(gg), dim3(256), sm, st, xb, wb, swg, T, c.hidden, E, stride, lg);
    }
  } else {
    dim3 g1((E1 + kRBM - 1) / kRBM, (T + kRBN - 1) / kRBN);
    if (c.dtype == MOE_BF16)
      launch_pdl(router_logits_kernel<MOE_BF16>, dim3(g1), dim3(256), 0, st, xb, wb, swg, T, c.hidden, E, stride, lg);
    else
      launch_pdl(router_logits_kernel<MOE_F16>, dim3(g1), dim3(256), 0, st, xb, wb, swg, T, c.hidden, E, stride, lg);
  }
  if (moe_status_t s = check_launch("router_logits_kernel")) return s;
  if (nsplit_out) {  // the caller ranks (fused with its grouping)
    *nsplit_out = nsplit;
    stat_kernels(1);
    return MOE_OK;
  }
  // The logits rows are laid out with stride E1 only when the gate column exists.
  dim3 g2((T + 7) / 8);
  if (E <= 256)
    launch_pdl(router_topk_kernel<8>, dim3(g2), dim3(256), 0, st, lg, reinterpret_cast<const float*>(ws + L.r_part),
               nsplit, T, E, stride, c.top_k, c.norm_topk, ids, w, logits_out, cnt, rank);
  else
    launch_pdl(router_topk_kernel<32>, dim3(g2), dim3(256), 0, st, lg, static_cast<const float*>(nullptr), 0, T, E,
               stride, c.top_k, c.norm_topk, ids, w, logits_out, cnt, rank);
  if (moe_status_t s = check_launch("router_topk_kernel")) return s;
  stat_kernels(2);
  return MOE_OK;
}

}  // namespace moe
