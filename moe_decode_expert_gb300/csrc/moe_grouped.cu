// moe_grouped.cu — the MoE block for T > 1 tokens, grouped per expert.
//
// "Decode throughput analysis report", code-level profiling section: with
// T >= 2 the pages' code fell into a prefill path that pulled the unique
// expert ids to the host and looped over experts in Python; their fix
// flattened the T*k (token, expert) pairs into batched products, and their
// next step is a grouped GEMM.  Here the grouping happens on the device, with
// no host synchronisation:
//   group    counting sort of the T*k pairs by expert id (plus T pairs of
//            the shared expert, filed as expert E), tile list of up to kTN
//            pairs of one expert;
//   w13      per (tile, block of gate/up pairs): the expert's W13 rows are
//            streamed once per tile and dotted with the tile's tokens,
//            SiLU(gate)*up -> act[pair] (fp32);
//   w2       per (tile, block of output rows): y[pair, h] = weight(pair) *
//            W2[e, h, :] . act[pair] (routing weight, or the shared gate);
//   combine  out[t] = sum_j y[t*k + j] (+ y[shared pair of t]) in slot order.
// Every output element is produced by one fixed sequence of fp32 operations,
// so results do not depend on the order in which pairs were filed.

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_stages.cuh"

namespace moe {

constexpr int kGThreads = 256;
constexpr int kGWarps = kGThreads / 32;
constexpr int kPB = 32;           // gate/up pairs per w13 work item
constexpr int kHB = 64;           // output rows per w2 work item

// ------------------------------------------------------------- grouping
// One CTA of 1024 threads.  counts/offsets/tiles live in the workspace.
__global__ void __launch_bounds__(1024) group_kernel(const int32_t* ids, int T, int k, int E,
                                                     int has_shared, int32_t* counts_out,
                                                     int32_t* offsets, int32_t* perm, int32_t* tiles,
                                                     int write_tiles, Control* ctrl) {
  pdl_launch_dependents();  // let the next kernel on the stream launch early
  pdl_wait();               // inputs written by the previous kernel are visible
  group_stage(ids, T, k, E, has_shared, counts_out, offsets, perm, tiles, write_tiles, ctrl);
}

// Token of pair p (routed pairs t*k + j, then shared pairs T*k + t).
__device__ __forceinline__ int pair_token(int p, int T, int k) { return p < T * k ? p / k : p - T * k; }

// ----------------------------------------------------------- W13 + SiLU
template <int DT>
__global__ void __launch_bounds__(kGThreads) grouped_w13_kernel(
    const uint8_t* x, const uint8_t* w13, const uint8_t* sw13,
    const int32_t* counts, const int32_t* offsets,
    const int32_t* perm, const int32_t* tiles, int T, int H, int E, int k,
    int I, int Is, int act_stride, float* __restrict__ act) {
  pdl_launch_dependents();  // let the next kernel on the stream launch early
  pdl_wait();               // inputs written by the previous kernel are visible
  extern __shared__ __align__(16) float xs[];   // [kTN][H] fp32
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = counts[E + 1];
  const int Imax = I > Is ? I : Is;
  const int npb = (Imax + kPB - 1) / kPB;
  const size_t rowb = static_cast<size_t>(H) * 2;
  const int nch = H >> 3;
  for (int item = blockIdx.x; item < n_tiles * npb; item += gridDim.x) {
    const int tile = item / npb, pb = item - tile * npb;
    const int e = tiles[2 * tile], start = tiles[2 * tile + 1];
    const int seg_end = offsets[e] + counts[e];
    const int nt = min(kTN, seg_end - start);
    const int ie = e == E ? Is : I;
    if (pb * kPB >= ie) continue;
    __syncthreads();  // previous item's readers of xs are done
    for (int idx = threadIdx.x; idx < nt * nch; idx += kGThreads) {
      const int r = idx / nch, c = idx - r * nch;
      const int t = pair_token(perm[start + r], T, k);
      float f[8];
      unpack8<DT>(ld_nc16(x + static_cast<size_t>(t) * rowb + 16 * static_cast<size_t>(c)), f);
      float4* d = reinterpret_cast<float4*>(xs + static_cast<size_t>(r) * H + 8 * c);
      d[0] = make_float4(f[0], f[1], f[2], f[3]);
      d[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
    __syncthreads();
    const uint8_t* base = e == E ? sw13 : w13 + static_cast<size_t>(e) * 2 * I * rowb;
    for (int i = pb * kPB + warp; i < min(ie, (pb + 1) * kPB); i += kGWarps) {
      const uint8_t* g_row = base + static_cast<size_t>(i) * rowb;
      const uint8_t* u_row = base + static_cast<size_t>(ie + i) * rowb;
      float ag[kTN], au[kTN];
#pragma unroll
      for (int r = 0; r < kTN; ++r) { ag[r] = 0.f; au[r] = 0.f; }
      for (int c = lane; c < nch; c += 32) {
        float fg[8], fu[8];
        unpack8<DT>(ld_stream16(g_row + 16 * static_cast<size_t>(c)), fg);
        unpack8<DT>(ld_stream16(u_row + 16 * static_cast<size_t>(c)), fu);
#pragma unroll
        for (int r = 0; r < kTN; ++r) {
          if (r < nt) {
            const float4 xa = reinterpret_cast<const float4*>(xs + static_cast<size_t>(r) * H)[2 * c];
            const float4 xb = reinterpret_cast<const float4*>(xs + static_cast<size_t>(r) * H)[2 * c + 1];
            const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              ag[r] = fmaf(fg[q], xv[q], ag[r]);
              au[r] = fmaf(fu[q], xv[q], au[r]);
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kTN; ++r) {
        const float g = warp_sum(ag[r]);
        const float u = warp_sum(au[r]);
        if (lane == 0 && r < nt) act[static_cast<size_t>(perm[start + r]) * act_stride + i] = silu_f(g) * u;
      }
    }
  }
}

// ------------------------------------------------------ W2 + pair weight
template <int DT>
__global__ void __launch_bounds__(kGThreads) grouped_w2_kernel(
    const uint8_t* w2, const uint8_t* sw2, const int32_t* counts,
    const int32_t* offsets, const int32_t* perm,
    const int32_t* tiles, const float* topk_w,
    const float* gate_logits, int gate_stride, int has_gate, int T, int H, int E, int k,
    int I, int Is, int act_stride, const float* act, float* __restrict__ y) {
  pdl_launch_dependents();  // let the next kernel on the stream launch early
  pdl_wait();               // inputs written by the previous kernel are visible
  extern __shared__ __align__(16) float as[];   // [kTN][Imax] fp32
  __shared__ float s_wt[kTN];
  __shared__ int s_pair[kTN];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = counts[E + 1];
  const int nhb = (H + kHB - 1) / kHB;
  for (int item = blockIdx.x; item < n_tiles * nhb; item += gridDim.x) {
    const int tile = item / nhb, hb = item - tile * nhb;
    const int e = tiles[2 * tile], start = tiles[2 * tile + 1];
    const int seg_end = offsets[e] + counts[e];
    const int nt = min(kTN, seg_end - start);
    const int ie = e == E ? Is : I;
    __syncthreads();
    if (threadIdx.x < nt) {
      const int p = perm[start + threadIdx.x];
      s_pair[threadIdx.x] = p;
      float wt;
      if (p < T * k) wt = topk_w[p];
      else wt = has_gate ? sigmoid_f(gate_logits[static_cast<size_t>(p - T * k) * gate_stride + E]) : 1.0f;
      s_wt[threadIdx.x] = wt;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < nt * (ie >> 2); idx += kGThreads) {
      const int r = idx / (ie >> 2), c = idx - r * (ie >> 2);
      reinterpret_cast<float4*>(as + static_cast<size_t>(r) * ie)[c] =
          reinterpret_cast<const float4*>(act + static_cast<size_t>(s_pair[r]) * act_stride)[c];
    }
    __syncthreads();
    const uint8_t* base = e == E ? sw2 : w2 + static_cast<size_t>(e) * H * I * 2;
    const int nch = ie >> 3;
    for (int h = hb * kHB + warp; h < min(H, (hb + 1) * kHB); h += kGWarps) {
      const uint8_t* row = base + static_cast<size_t>(h) * ie * 2;
      float acc[kTN];
#pragma unroll
      for (int r = 0; r < kTN; ++r) acc[r] = 0.f;
      for (int c = lane; c < nch; c += 32) {
        float f[8];
        unpack8<DT>(ld_stream16(row + 16 * static_cast<size_t>(c)), f);
#pragma unroll
        for (int r = 0; r < kTN; ++r) {
          if (r < nt) {
            const float4 xa = reinterpret_cast<const float4*>(as + static_cast<size_t>(r) * ie)[2 * c];
            const float4 xb = reinterpret_cast<const float4*>(as + static_cast<size_t>(r) * ie)[2 * c + 1];
            const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[r] = fmaf(f[q], xv[q], acc[r]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kTN; ++r) {
        const float s = warp_sum(acc[r]);
        if (lane == 0 && r < nt) y[static_cast<size_t>(s_pair[r]) * H + h] = s_wt[r] * s;
      }
    }
  }
}

// ---------------------------------------------------------------- combine
__global__ void __launch_bounds__(256) combine_kernel(const float* y, int T, int H, int k,
                                                      int has_shared, void* out, int out_dtype,
                                                      const uint16_t* xres, int x_dtype) {
  pdl_launch_dependents();  // let the next kernel on the stream launch early
  pdl_wait();               // inputs written by the previous kernel are visible
  // grid (ceil(H/4 / 256), T): four consecutive outputs of token blockIdx.y per
  // thread (H % 8 == 0); the sum runs in slot order, then the shared part
  const int H4 = H >> 2;
  const int h4 = blockIdx.x * 256 + threadIdx.x;
  const int t = blockIdx.y;
  if (h4 >= H4 || t >= T) return;
  const float4* y4 = reinterpret_cast<const float4*>(y);
  const int nk = k + (has_shared ? 1 : 0);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < nk; j0 += 8) {  // eight slot loads in flight, then add in order
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u;
      if (j < nk) {
        const size_t row = j < k ? static_cast<size_t>(t) * k + j : static_cast<size_t>(T) * k + t;
        v[u] = y4[row * H4 + h4];
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (j0 + u < nk) { acc.x += v[u].x; acc.y += v[u].y; acc.z += v[u].z; acc.w += v[u].w; }
  }
  const size_t o = static_cast<size_t>(t) * H + 4 * h4;
  if (xres) {  // residual add (MOE_FLAG_RESIDUAL): out = x + block(x)
    const uint2 r = *reinterpret_cast<const uint2*>(xres + o);
    const float2 a = x_dtype == MOE_BF16 ? unpack2<MOE_BF16>(r.x) : unpack2<MOE_F16>(r.x);
    const float2 b = x_dtype == MOE_BF16 ? unpack2<MOE_BF16>(r.y) : unpack2<MOE_F16>(r.y);
    acc.x += a.x; acc.y += a.y; acc.z += b.x; acc.w += b.y;
  }
  store_out(out, o, acc.x, out_dtype);
  store_out(out, o + 1, acc.y, out_dtype);
  store_out(out, o + 2, acc.z, out_dtype);
  store_out(out, o + 3, acc.w, out_dtype);
}

moe_status_t launch_grouped(const moe_cfg_t& c, const BlockPtrs& p, uint8_t* ws, const WsLayout& L,
                            int32_t T, cudaStream_t st) {
  const int H = c.hidden, E = c.n_experts, k = c.top_k, I = c.inter, Is = c.shared_inter;
  Control* ctrl = reinterpret_cast<Control*>(ws + L.ctrl);
  const bool use_tc = !(c.flags & MOE_FLAG_GROUPED_SIMT) && L.tc_n > 0 && tc_path_supported(c);
  // small batches on the tensor-core path: ranking, grouping and tile lists in
  // one single-CTA launch, a warp per token
  const bool fused = use_tc && T <= kRouteGroupMaxT && E <= 256;
  // larger batches on the tensor-core path: the top-k kernel ranks each pair
  // within its expert, and the pass launcher files them (no counting sort)
  const bool ranked = use_tc && !fused;
  int nsplit = -1;
  if (moe_status_t s = launch_router(c, p.x, p.router_w, p.shared_gate_w, T, p.topk_ids, p.topk_w,
                                     nullptr, ws, L, st, fused ? &nsplit : nullptr,
                                     ranked ? reinterpret_cast<int32_t*>(ws + L.tc_cnt) : nullptr,
                                     ranked ? reinterpret_cast<int32_t*>(ws + L.tc_rank) : nullptr))
    return s;
  int32_t* counts = reinterpret_cast<int32_t*>(ws + L.g_counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + L.g_offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(ws + L.g_perm);
  int32_t* tiles = reinterpret_cast<int32_t*>(ws + L.g_tiles);
  float* act = reinterpret_cast<float*>(ws + L.g_act);
  float* y = reinterpret_cast<float*>(ws + L.g_y);
  const float* glog = reinterpret_cast<const float*>(ws + L.r_logits);
  const int gate_stride = c.has_shared_gate ? E + 1 : E;
  const int Imax = I > Is ? I : Is;

  if (!fused && !ranked) {
    launch_pdl(group_kernel, dim3(1), dim3(1024), 0, st, p.topk_ids, T, k, E, Is > 0, counts, offsets, perm, tiles,
               use_tc ? 0 : 1, ctrl);
    if (moe_status_t s = check_launch("group_kernel")) return s;
    stat_kernels(1);
  }

  const int sms = sm_count();
  if ((c.flags & MOE_FLAG_GROUPED_TC) && !use_tc)
    return set_error(MOE_ERR_UNSUPPORTED, "grouped: the tensor-core path needs H %% 128 == 0, "
                                          "I and Is multiples of 64 and the TMA encoder");
  if (use_tc) {
    if (moe_status_t s = launch_tc_passes(c, p, ws, L, T, fused ? nsplit : -1, st)) return s;
    stat_grouped_tc();
  } else {
    const size_t smem13 = static_cast<size_t>(kTN) * H * 4;
    const size_t smem2 = static_cast<size_t>(kTN) * Imax * 4;
    if (smem13 > 227 * 1024 || smem2 > 227 * 1024)
      return set_error(MOE_ERR_UNSUPPORTED, "grouped: hidden=%d or inter=%d too large for one tile", H, Imax);
    const int npb = (Imax + kPB - 1) / kPB;
    const int nhb = (H + kHB - 1) / kHB;
    const long long items13 = L.max_tiles * npb, items2 = L.max_tiles * nhb;
    const int g13 = static_cast<int>(items13 < sms * 8LL ? items13 : sms * 8LL);
    const int g2 = static_cast<int>(items2 < sms * 8LL ? items2 : sms * 8LL);
    const uint8_t* x = static_cast<const uint8_t*>(p.x);
    if (c.dtype == MOE_BF16) {
      raise_smem_limit(grouped_w13_kernel<MOE_BF16>, smem13);
      launch_pdl(grouped_w13_kernel<MOE_BF16>, dim3(g13), dim3(kGThreads), smem13, st, 
          x, static_cast<const uint8_t*>(p.w13), static_cast<const uint8_t*>(p.shared_w13), counts, offsets,
          perm, tiles, T, H, E, k, I, Is, Imax, act);
    } else {
      raise_smem_limit(grouped_w13_kernel<MOE_F16>, smem13);
      launch_pdl(grouped_w13_kernel<MOE_F16>, dim3(g13), dim3(kGThreads), smem13, st, 
          x, static_cast<const uint8_t*>(p.w13), static_cast<const uint8_t*>(p.shared_w13), counts, offsets,
          perm, tiles, T, H, E, k, I, Is, Imax, act);
    }
    if (moe_status_t s = check_launch("grouped_w13_kernel")) return s;
    if (c.dtype == MOE_BF16) {
      raise_smem_limit(grouped_w2_kernel<MOE_BF16>, smem2);
      launch_pdl(grouped_w2_kernel<MOE_BF16>, dim3(g2), dim3(kGThreads), smem2, st, 
          static_cast<const uint8_t*>(p.w2), static_cast<const uint8_t*>(p.shared_w2), counts, offsets, perm,
          tiles, p.topk_w, glog, gate_stride, c.has_shared_gate, T, H, E, k, I, Is, Imax, act, y);
    } else {
      raise_smem_limit(grouped_w2_kernel<MOE_F16>, smem2);
      launch_pdl(grouped_w2_kernel<MOE_F16>, dim3(g2), dim3(kGThreads), smem2, st, 
          static_cast<const uint8_t*>(p.w2), static_cast<const uint8_t*>(p.shared_w2), counts, offsets, perm,
          tiles, p.topk_w, glog, gate_stride, c.has_shared_gate, T, H, E, k, I, Is, Imax, act, y);
    }
    if (moe_status_t s = check_launch("grouped_w2_kernel")) return s;
    stat_kernels(2);
  }
  const uint16_t* xres = (c.flags & MOE_FLAG_RESIDUAL) ? static_cast<const uint16_t*>(p.x) : nullptr;
  launch_pdl(combine_kernel, dim3((H / 4 + 255) / 256, T), dim3(256), 0, st, y, T, H, k, Is > 0, p.out,
             c.out_dtype, xres, c.dtype);
  if (moe_status_t s = check_launch("combine_kernel")) return s;
  stat_kernels(1);
  return MOE_OK;
}

}  // namespace moe
