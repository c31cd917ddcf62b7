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

namespace moe {

constexpr int kRBM = 64;   // router rows (experts) per CTA tile
constexpr int kRBN = 64;   // tokens per CTA tile
constexpr int kRBK = 32;   // hidden elements per k-step

template <int DT>
__global__ void __launch_bounds__(256) router_logits_kernel(const uint8_t* __restrict__ x,
                                                            const uint8_t* __restrict__ wr,
                                                            const uint8_t* __restrict__ swg, int T,
                                                            int H, int E, int E1, float* __restrict__ logits) {
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

// One warp per token: rank, weights, outputs.
template <int MAXM>
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ logits, int T, int E,
                                                          int E1, int k, int norm_topk, int32_t* ids,
                                                          float* w, float* logits_out) {
  __shared__ int s_ids[8][32];
  __shared__ float s_sel[8][32];
  __shared__ float s_w[8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const float* row = logits + static_cast<size_t>(t) * E1;
  warp_topk<MAXM>(row, E, k, s_ids[warp], s_sel[warp]);
  __syncwarp();
  warp_routing_weights(row, E, s_sel[warp], k, norm_topk, s_w[warp]);
  __syncwarp();
  if (lane < k) {
    ids[static_cast<size_t>(t) * k + lane] = s_ids[warp][lane];
    w[static_cast<size_t>(t) * k + lane] = s_w[warp][lane];
  }
  if (logits_out)
    for (int e = lane; e < E; e += 32) logits_out[static_cast<size_t>(t) * E + e] = row[e];
}

moe_status_t launch_router(const moe_cfg_t& c, const void* x, const void* router_w,
                           const void* shared_gate_w, int32_t T, int32_t* ids, float* w,
                           float* logits_out, uint8_t* ws, const WsLayout& L, cudaStream_t st) {
  const int E = c.n_experts;
  const int E1 = E + 1;
  float* lg = reinterpret_cast<float*>(ws + L.r_logits);
  const uint8_t* swg = c.has_shared_gate ? static_cast<const uint8_t*>(shared_gate_w) : nullptr;
  dim3 g1((E1 + kRBM - 1) / kRBM, (T + kRBN - 1) / kRBN);
  if (c.dtype == MOE_BF16)
    router_logits_kernel<MOE_BF16><<<g1, 256, 0, st>>>(static_cast<const uint8_t*>(x),
                                                       static_cast<const uint8_t*>(router_w), swg, T,
                                                       c.hidden, E, swg ? E1 : E, lg);
  else
    router_logits_kernel<MOE_F16><<<g1, 256, 0, st>>>(static_cast<const uint8_t*>(x),
                                                      static_cast<const uint8_t*>(router_w), swg, T,
                                                      c.hidden, E, swg ? E1 : E, lg);
  if (moe_status_t s = check_launch("router_logits_kernel")) return s;
  // The logits rows are laid out with stride E1 only when the gate column exists.
  const int stride = swg ? E1 : E;
  dim3 g2((T + 7) / 8);
  if (E <= 256)
    router_topk_kernel<8><<<g2, 256, 0, st>>>(lg, T, E, stride, c.top_k, c.norm_topk, ids, w, logits_out);
  else
    router_topk_kernel<32><<<g2, 256, 0, st>>>(lg, T, E, stride, c.top_k, c.norm_topk, ids, w, logits_out);
  if (moe_status_t s = check_launch("router_topk_kernel")) return s;
  stat_kernels(2);
  return MOE_OK;
}

}  // namespace moe
