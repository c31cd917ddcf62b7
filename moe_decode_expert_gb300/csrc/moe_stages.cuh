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
  if (tid == 0) {
    *n13 = tot13;
    *n2 = tot2;
    n13[2] = 0;  // the two passes' dynamic tile counters (n13[0..3] is the schedule block)
    n13[3] = 0;
  }
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

// Small batches (T*k routed pairs plus the shared expert's entry at most
// kWarpGroupPairs): the grouping of the pairs by expert by one warp, then the
// tile lists by every thread after one CTA barrier (the tile-list kernels and
// the passes read only perm and the lists).  Pair p (routed: token p / k, slot
// p % k) gets the unique key (expert << 16) | p; its rank among all keys (rank
// counting over shared memory) is its sorted position, so each expert's pairs
// are filed in pair order.  Runs of equal experts in sorted order are the
// distinct experts, in ascending order, followed by the shared expert (index
// E, its T pairs in token order after the routed ones): the same lists the
// CTA-wide grouping and scheduling stages build.  flat_ids: the [T, k] ids in
// shared memory.  Called by every thread of the CTA.
constexpr int kWarpGroupPairs = 128;
struct WarpGroupScratch {
  uint32_t key[kWarpGroupPairs];
  uint32_t sorted[kWarpGroupPairs];
  int ue[kWarpGroupPairs + 1], upos[kWarpGroupPairs + 2], pre13[kWarpGroupPairs + 2], pre2[kWarpGroupPairs + 2];
  int nall, tot13, tot2;
};
__device__ __forceinline__ void small_group_schedule(const int32_t* flat_ids, int T, int k, int E, int has_shared,
                                                     int32_t* perm, Control* ctrl, int I, int Is, int H, int N,
                                                     int mt13, int mt2, int32_t* n13, int32_t* n2, TcTile* t13,
                                                     TcTile* t2) {
  constexpr int KPL = kWarpGroupPairs / 32;  // pairs per lane
  __shared__ __align__(16) WarpGroupScratch sc;
  const int tid = threadIdx.x, lane = tid & 31;
  const int np = T * k;  // np + has_shared <= kWarpGroupPairs (checked by the caller)
  if (tid < 32) {
    uint32_t key[KPL];
#pragma unroll
    for (int r = 0; r < KPL; ++r) {
      const int p = lane + 32 * r;
      key[r] = 0xffffffffu;
      if (p < np) {
        int e = flat_ids[p];
        if (e < 0 || e >= E) {
          report_error(ctrl, kDevBadExpert, static_cast<uint32_t>(p));
          e = 0;
        }
        key[r] = (static_cast<uint32_t>(e) << 16) | static_cast<uint32_t>(p);
      }
      sc.key[p] = key[r];
    }
    __syncwarp();
    int rk[KPL];
#pragma unroll
    for (int r = 0; r < KPL; ++r) rk[r] = 0;
    for (int j = 0; j < np; j += 4) {  // keys past np are all-ones: never smaller
      const uint4 kk = *reinterpret_cast<const uint4*>(sc.key + j);  // broadcast
#pragma unroll
      for (int r = 0; r < KPL; ++r)
        rk[r] += (kk.x < key[r]) + (kk.y < key[r]) + (kk.z < key[r]) + (kk.w < key[r]);
    }
#pragma unroll
    for (int r = 0; r < KPL; ++r)
      if (lane + 32 * r < np) {
        perm[rk[r]] = static_cast<int32_t>(key[r] & 0xffffu);
        sc.sorted[rk[r]] = key[r];
      }
    if (has_shared)
      for (int t = lane; t < T; t += 32) perm[np + t] = np + t;
    __syncwarp();
    // distinct experts: sorted positions where the expert changes
    int nu = 0;
#pragma unroll
    for (int r = 0; r < KPL; ++r) {
      const int pos = lane + 32 * r;
      const bool start = pos < np && (pos == 0 || (sc.sorted[pos] >> 16) != (sc.sorted[pos - 1] >> 16));
      const uint32_t m = __ballot_sync(0xffffffffu, start);
      if (start) {
        const int u = nu + __popc(m & ((1u << lane) - 1u));
        sc.ue[u] = static_cast<int>(sc.sorted[pos] >> 16);
        sc.upos[u] = pos;
      }
      nu += __popc(m);
    }
    if (lane == 0) {
      if (has_shared) {
        sc.ue[nu] = E;
        sc.upos[nu] = np;
      }
      sc.upos[nu + (has_shared ? 1 : 0)] = np + (has_shared ? T : 0);  // end of the last run
    }
    __syncwarp();
    const int nall = nu + (has_shared ? 1 : 0);
    // tiles of each distinct expert, then an exclusive scan (KPL entries per lane)
    int a13[KPL], a2[KPL], s13 = 0, s2 = 0;
#pragma unroll
    for (int r = 0; r < KPL; ++r) {
      const int u = KPL * lane + r;
      a13[r] = a2[r] = 0;
      if (u < nall) {
        const int e = sc.ue[u], cnt = sc.upos[u + 1] - sc.upos[u];
        const int ie = e == E ? Is : I;
        const int nt = (cnt + N - 1) / N;
        a13[r] = ie > 0 ? nt * ((ie / 64 + mt13 - 1) / mt13) : 0;
        a2[r] = ie > 0 ? nt * ((H / 128 + mt2 - 1) / mt2) : 0;
      }
      s13 += a13[r];
      s2 += a2[r];
    }
    int i13 = s13, i2 = s2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y13 = __shfl_up_sync(0xffffffffu, i13, o), y2 = __shfl_up_sync(0xffffffffu, i2, o);
      if (lane >= o) { i13 += y13; i2 += y2; }
    }
    int b13 = i13 - s13, b2 = i2 - s2;
#pragma unroll
    for (int r = 0; r < KPL; ++r) {
      const int u = KPL * lane + r;
      if (u < nall) {
        sc.pre13[u] = b13;
        sc.pre2[u] = b2;
      }
      b13 += a13[r];
      b2 += a2[r];
    }
    if (lane == 31) {
      sc.nall = nall;
      sc.tot13 = i13;
      sc.tot2 = i2;
      *n13 = i13;
      *n2 = i2;
      n13[2] = 0;  // the two passes' dynamic tile counters
      n13[3] = 0;
    }
  }
  __syncthreads();
  // tile i belongs to the last distinct expert whose first tile index is <= i
  const int nall = sc.nall, tot13 = sc.tot13, tot2 = sc.tot2;
  for (int i = tid; i < tot13 + tot2; i += blockDim.x) {
    const bool second = i >= tot13;
    const int ii = second ? i - tot13 : i;
    const int* pre = second ? sc.pre2 : sc.pre13;
    int lo = 0, hi = nall - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= ii) lo = mid; else hi = mid - 1;
    }
    const int e = sc.ue[lo];
    const int ie = e == E ? Is : I;
    const int per_n = second ? (H / 128 + mt2 - 1) / mt2 : (ie / 64 + mt13 - 1) / mt13;
    const int j = (ii - pre[lo]) / per_n, mm = (ii - pre[lo]) - j * per_n;
    const int cnt = sc.upos[lo + 1] - sc.upos[lo];
    const TcTile tl{e, mm, sc.upos[lo] + j * N, min(N, cnt - j * N)};
    if (second) t2[ii] = tl; else t13[ii] = tl;
  }
}

}  // namespace moe
