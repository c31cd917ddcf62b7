// moe_stages.cuh — device stages shared by the standalone routing/grouping
// kernels and the fused small-batch kernel: one token's top-k, the counting
// sort of (token, slot) pairs by expert, and the tensor-core tile lists.
#pragma once

#include "moe_common.cuh"

namespace moe {

constexpr int kTN = 8;  // pairs (tokens) per tile of the CUDA-core grouped kernels
constexpr int kRouteGroupMaxT = 32;  // tokens of the single-CTA ranking + grouping kernel (a warp each)

struct TcTile {
  int32_t e;     // expert id, E = shared expert
  int32_t m;     // M-tile index within the expert
  int32_t pos0;  // first sorted pair position of the N-tile
  int32_t n;     // valid tokens in the tile
};

// Router logits from its split partial sums part[s][t][e] (flat index
// q = t * E1 + e, split stride T * E1): v[c] = sum over s, in split order, of
// part[s][q0 + step * c] for q0 + step * c < limit (0 otherwise), with
// kSumCols x 8 loads in flight per thread.
constexpr int kSumCols = 3;
__device__ __forceinline__ void sum_splits(const float* part, int nsplit, size_t stride, int q0,
                                           int step, int limit, float (&v)[kSumCols]) {
#pragma unroll
  for (int c = 0; c < kSumCols; ++c) v[c] = 0.0f;
  for (int s0 = 0; s0 < nsplit; s0 += 8) {
    float pv[kSumCols][8];
#pragma unroll
    for (int c = 0; c < kSumCols; ++c)
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int q = q0 + step * c;
        const bool in = q < limit && s0 + u < nsplit;
        pv[c][u] = in ? part[static_cast<size_t>(s0 + u) * stride + q] : 0.0f;
      }
    // adding +0 for a missing split leaves the sum unchanged (it is never -0)
#pragma unroll
    for (int c = 0; c < kSumCols; ++c)
#pragma unroll
      for (int u = 0; u < 8; ++u) v[c] += pv[c][u];
  }
}

// One token's ranking, routing weights and outputs (called by one full warp;
// s_* are this warp's scratch rows in shared memory).  With nsplit > 0 the
// logits arrive as nsplit partial sums part[s][t][e] (router_mma_kernel):
// they are added in split order, stored into `logits` (the [T, E1] buffer
// later kernels read) and ranked from s_row.
template <int MAXM>
__device__ __forceinline__ void topk_token_stage(float* logits, const float* part,
                                                 int nsplit, int t, int T, int E, int E1, int k, int norm_topk,
                                                 int32_t* ids, float* w, float* logits_out, int* s_ids,
                                                 float* s_sel, float* s_w, float* s_row) {
  const int lane = threadIdx.x & 31;
  const float* row = logits + static_cast<size_t>(t) * E1;
  if constexpr (MAXM == 8) {
    if (nsplit > 0) {
      for (int e0 = lane; e0 < E1; e0 += 32 * kSumCols) {
        float v[kSumCols];
        sum_splits(part, nsplit, static_cast<size_t>(T) * E1, t * E1 + e0, 32, t * E1 + E1, v);
#pragma unroll
        for (int c = 0; c < kSumCols; ++c) {
          const int e = e0 + 32 * c;
          if (e < E1) {
            s_row[e] = v[c];
            logits[static_cast<size_t>(t) * E1 + e] = v[c];
          }
        }
      }
      __syncwarp();
      row = s_row;
    }
  }
  if constexpr (MAXM == 8) warp_topk_sorted8(row, E, k, s_ids, s_sel);
  else warp_topk<MAXM>(row, E, k, s_ids, s_sel);
  __syncwarp();
  warp_routing_weights(row, E, s_sel, k, norm_topk, s_w);
  __syncwarp();
  if (lane < k) {
    ids[static_cast<size_t>(t) * k + lane] = s_ids[lane];
    w[static_cast<size_t>(t) * k + lane] = s_w[lane];
  }
  if (logits_out)
    for (int e = lane; e < E; e += 32) logits_out[static_cast<size_t>(t) * E + e] = row[e];
}

__device__ __forceinline__ void group_stage(const int32_t* ids, int T, int k, int E,
                                                     int has_shared, int32_t* counts_out,
                                                     int32_t* offsets, int32_t* perm, int32_t* tiles,
                                                     int write_tiles, Control* ctrl,
                                                     int32_t* s_counts = nullptr, int32_t* s_offsets = nullptr) {
  __shared__ int32_t cnt[1025 + 1];
  __shared__ int32_t cur[1025 + 1];
  __shared__ int32_t tcnt[1025 + 1];
  __shared__ int32_t wsum[32];
  const int tid = threadIdx.x;
  const int n = E + 1;  // experts + the shared expert
  for (int e = tid; e < n; e += 1024) cnt[e] = 0;
  __syncthreads();
  const int np = T * k;
  for (int base = tid; base < np; base += 1024 * 8) {  // 8 id loads in flight per thread
    int ev[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) ev[u] = base + 1024 * u < np ? ids[base + 1024 * u] : -2;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = ev[u];
      if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
      else if (e != -2) report_error(ctrl, kDevBadExpert, static_cast<uint32_t>(base + 1024 * u));
    }
  }
  if (tid == 0) cnt[E] = has_shared ? T : 0;
  __syncthreads();

  // Exclusive scans of pair counts and tile counts (two elements per thread at most).
  const int lane = tid & 31, warp = tid >> 5;
  int c0 = 0, c1 = 0, t0 = 0, t1 = 0;
  const int e0 = 2 * tid, e1 = 2 * tid + 1;
  if (e0 < n) { c0 = cnt[e0]; t0 = (c0 + kTN - 1) / kTN; }
  if (e1 < n) { c1 = cnt[e1]; t1 = (c1 + kTN - 1) / kTN; }
  // pack pair and tile sums into one 64-bit scan value
  unsigned long long v = (static_cast<unsigned long long>(c0 + c1) << 32) | static_cast<unsigned>(t0 + t1);
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  __shared__ unsigned long long wtot[32];
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    unsigned long long s = wtot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    wtot[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const unsigned long long before = incl - v + (warp ? wtot[warp - 1] : 0ull);
  const int pb = static_cast<int>(before >> 32), tb = static_cast<int>(before & 0xffffffffu);
  if (e0 < n) { cur[e0] = pb; tcnt[e0] = tb; }
  if (e1 < n) { cur[e1] = pb + c0; tcnt[e1] = tb + t0; }
  __syncthreads();
  (void)wsum;
  for (int e = tid; e < n; e += 1024) {
    offsets[e] = cur[e];
    counts_out[e] = cnt[e];
    if (s_offsets) {  // copies for a later stage of the same CTA
      s_offsets[e] = cur[e];
      s_counts[e] = cnt[e];
    }
  }
  const unsigned long long tot = wtot[31];
  const int n_tiles = static_cast<int>(tot & 0xffffffffu);
  if (tid == 0) {
    offsets[n] = static_cast<int>(tot >> 32);
    counts_out[n] = n_tiles;  // number of tiles
  }
  if (write_tiles) {
    // tile i belongs to the last expert whose first tile index is <= i
    for (int i = tid; i < n_tiles; i += 1024) {
      int lo = 0, hi = n - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tcnt[mid] <= i) lo = mid; else hi = mid - 1;
      }
      tiles[2 * i] = lo;
      tiles[2 * i + 1] = cur[lo] + (i - tcnt[lo]) * kTN;
    }
  }
  __syncthreads();
  // File routed pairs (any order within an expert) and the shared pairs (in token order).
  for (int base = tid; base < np; base += 1024 * 8) {
    int ev[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) ev[u] = base + 1024 * u < np ? ids[base + 1024 * u] : -2;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = ev[u];
      if (e >= 0 && e < E) perm[atomicAdd(&cur[e], 1)] = base + 1024 * u;
    }
  }
  if (has_shared)
    for (int t = tid; t < T; t += 1024) perm[cur[E] + t] = np + t;
}

__device__ __forceinline__ void schedule_stage(const int32_t* counts,
                                                           const int32_t* offsets, int E, int I,
                                                           int Is, int H, int N, int mt13, int mt2, int32_t* n13,
                                                           int32_t* n2, TcTile* t13, TcTile* t2) {
  __shared__ unsigned long long wtot[32];
  __shared__ int pre13[1026], pre2[1026];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = E + 1;
  // tiles of each expert (two experts per thread; n <= 1025)
  int a13[2] = {0, 0}, a2[2] = {0, 0};
  for (int s = 0; s < 2; ++s) {
    const int e = 2 * tid + s;
    if (e < n) {
      const int cnt = counts[e];
      const int ie = e == E ? Is : I;
      const int nt = (cnt + N - 1) / N;
      a13[s] = ie > 0 ? nt * ((ie / 64 + mt13 - 1) / mt13) : 0;
      a2[s] = ie > 0 ? nt * ((H / 128 + mt2 - 1) / mt2) : 0;
    }
  }
  unsigned long long v = (static_cast<unsigned long long>(a13[0] + a13[1]) << 32) | static_cast<unsigned>(a2[0] + a2[1]);
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long yv = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += yv;
  }
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    unsigned long long s = wtot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long yv = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += yv;
    }
    wtot[lane] = s;
  }
  __syncthreads();
  const unsigned long long before = incl - v + (warp ? wtot[warp - 1] : 0ull);
  const int b13 = static_cast<int>(before >> 32), b2 = static_cast<int>(before & 0xffffffffu);
  if (2 * tid < n) { pre13[2 * tid] = b13; pre2[2 * tid] = b2; }
  if (2 * tid + 1 < n) { pre13[2 * tid + 1] = b13 + a13[0]; pre2[2 * tid + 1] = b2 + a2[0]; }
  __syncthreads();
  const int tot13 = static_cast<int>(wtot[31] >> 32), tot2 = static_cast<int>(wtot[31] & 0xffffffffu);
  if (tid == 0) { *n13 = tot13; *n2 = tot2; }
  // Fill both lists in parallel: tile i belongs to the last expert whose first
  // tile index is <= i (experts without tiles share their successor's start).
  for (int i = tid; i < tot13 + tot2; i += 1024) {
    const bool second = i >= tot13;
    const int ii = second ? i - tot13 : i;
    const int* pre = second ? pre2 : pre13;
    int lo = 0, hi = n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= ii) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int ie = e == E ? Is : I;
    const int per_n = second ? (H / 128 + mt2 - 1) / mt2 : (ie / 64 + mt13 - 1) / mt13;  // M-groups per N-tile
    const int j = (ii - pre[e]) / per_n, mm = (ii - pre[e]) - j * per_n;
    const int cnt = counts[e];
    const TcTile tl{e, mm, offsets[e] + j * N, min(N, cnt - j * N)};
    if (second) t2[ii] = tl; else t13[ii] = tl;
  }
}

}  // namespace moe
